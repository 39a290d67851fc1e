// chunk_tc.cu -- the KDA chunked forward on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), for bf16 I/O with K = V = 128 and chunk C = 64.
//
// Two kernels share the chunk loop below.  The fused kernel keeps the fp32 state S (K x V)
// in TMEM and walks the chunks of a sequence in order: one CTA (16 warps) per (b, h), or,
// with more sequences than SMs, one CTA per SM taking (segment, sequence) work items and
// handing the state between segments (FusedSched).  The prep kernel of the split form runs
// P2-P5 for every (sequence, chunk) item in parallel and writes the state-independent
// operands for the carry kernel (chunk_carry.cu).  Per chunk:
//
//   P1  TMA: q, k, z tiles (64 x 128 bf16 each) and the v tile, on two mbarriers; the
//       next chunk's tiles are requested as soon as each slot is consumed (q, k, z in
//       P5, v after C3).
//   P2  gate g = -exp(A_log) softplus(z + dt_bias) and the in-chunk cumulative log decay
//       G (kdafix-2026-10-02 "Fix 1"; kda-adjoint-2026-10-01 sec. 2), and the pairs
//       inside 4-token blocks (exact pairwise exponential, CUDA cores); in the fused
//       kernel warps 8-15 do both for chunk n+1 while warps 0-7 do chunk n's C1-C3.
//   P3  decay-folded scores  A[t,i] = beta_t sum_c k_tc k_ic e^{G_tc - G_ic}  (i < t) and
//       M[t,i] = sum_c q_tc k_ic e^{G_tc - G_ic}  (i <= t).  e^{G_t - G_i} cannot be split
//       as e^{G_t} e^{-G_i} (e^{-G_i} overflows fp32 within a chunk when the decay is
//       strong), so pairs are grouped by the level of the binary tree over the 64 tokens
//       at which t and i part: at half-width h, t in the upper half and i in the lower half
//       of one 2h-block share the reference r = last token of the lower half, and
//       e^{G_t - G_i} = e^{G_t - G_r} e^{G_r - G_i} with both factors <= 1.  Levels
//       h = 32, 16, 8, 4 go two per tcgen05 GEMM (each level's upper k and q rows against
//       its lower k rows, tokens in rank order); an epilogue scatters them to A and M.
//   P4  T = (I + A)^{-1}: 16 x 16 diagonal blocks by forward substitution (fp32, CUDA
//       cores), then the block merges T_21 = -T_22 A_21 T_11 (16 -> 32 for both halves at
//       once, then 32 -> 64) as four small tcgen05 products with bf16 operands.
//   P5  W^T = (diag(beta) K Gamma)^T T^T and U^T = (diag(beta) V)^T T^T  (tcgen05).  The
//       fused kernel forms Q Gamma row-major (a K-major operand [t][c]) during the inverse's
//       merges, on the warps that read no merge product; the prep kernel puts (Q Gamma)^T
//       next to W^T in A1.
//   C1  D = S^T [W^T | (Q Gamma)^T] = [(W S)^T | (Q Gamma S)^T]  (M = 128 value channels,
//       N = 64 + 64, K = 128; S as bf16 operand), so that Delta = U - W S and the state's
//       share of the output come from one pass over S.  Before it, the fp32 state in TMEM is
//       scaled by Gamma_last (row c by e^{G_last,c}).
//   C2  from TMEM, one value channel per thread: Delta^T = U^T - (W S)^T.
//   C3  S += (K * e^{G_last - G})^T Delta   accumulated in TMEM in fp32 (the carry with a
//       single exponential of the log-space difference, kda-adjoint-2026-10-01 sections 2
//       and 5b), and (M Delta)^T onto (Q Gamma S)^T: o = scale (Q Gamma S + M Delta), which
//       is scale (Q' S + U') with Q' = Q Gamma - M W and U' = M U, goes out as bf16 during
//       the next chunk's inverse.  The new S becomes the bf16 operand under the next W/U GEMM.
//
// Operand layouts are the tcgen05 canonical 128-byte-swizzled layouts, either K-major
// (rows of 128 B along the contraction) or MN-major (rows of 128 B along M/N); both are
// written directly by the threads that produce them.  Every mbarrier and flag wait is
// bounded; on a timeout the CTA records it in g_kda_tc_timeout, releases its TMEM and exits.
#include <cuda.h>
#include <stddef.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "chunk_tiles.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace kda {

__device__ int g_kda_tc_timeout;

namespace {

using namespace tile;
constexpr int NT = 512;
constexpr float LOG2E = 1.4426950408889634f;

// ---- shared memory map (bytes from a 1024-byte aligned base)
constexpr uint32_t OFF_LVL = 0;                 // 64 KB multi-use region (see LV_*)
constexpr uint32_t OFF_G = 65536;               // 32 KB fp32 G[t][c]
constexpr uint32_t OFF_Q = OFF_G + 32768;       // 16 KB bf16 q tile, row-major [t][c]
constexpr uint32_t OFF_K = OFF_Q + 16384;       // 16 KB bf16 k tile
constexpr uint32_t OFF_V = OFF_K + 16384;       // 16 KB bf16 v tile, then K~
constexpr uint32_t OFF_A1 = OFF_V + 16384;      // 32 KB W^T | (prep kernel) (Q Gamma)^T, MN-major
constexpr uint32_t OFF_S = OFF_A1 + 32768;      // 32 KB S bf16, MN-major [c][v] (2 atoms)
constexpr uint32_t OFF_MISC = OFF_S + 32768;
// multi-use region, in order of use within a chunk
constexpr uint32_t LV_PA = 0;       // level pair A operand, K-major 128 rows (32 KB)   P3
constexpr uint32_t LV_PB = 32768;   // level pair B operand, K-major 64 rows (16 KB)    P3
constexpr uint32_t LV_AF = 0;       // A fp32 [t][i] (16 KB, swizzled; diagonal 16 x 16 blocks)  P3-P4
constexpr uint32_t LV_MB = 16384;   // M bf16 K-major [t][i] (8 KB)          P3-P5 (fused: -C3)
constexpr uint32_t LV_TB = 24576;   // T bf16 K-major [t][i] (8 KB)          P4-P5
constexpr uint32_t LV_Z = 49152;    // z tile of the NEXT chunk (16 KB)      P5-P2
constexpr uint32_t LV_GTF = 24576;  // fused kernel: the gate's warp totals (8 KB), in the T slot  window
constexpr uint32_t LV_QG = 0;       // fused kernel: Q Gamma bf16 K-major [t][c] (16 KB)  merges - C1
constexpr uint32_t LV_GTP = 32768;  // prep kernel: the gate's warp totals (8 KB)    S2
constexpr uint32_t LV_AB = 49152;   // A bf16 K-major [t][i] (8 KB), in the z slot         P3-P4
constexpr uint32_t LV_MG = 57344;   // merge products P, P' (8 KB), in the z slot            P4
constexpr uint32_t LV_DELTA = 32768;// Delta^T K-major [v][t] (16 KB)        C2-C3 (fused; M stays)
// K~ (K e^{G_last - G}, MN-major [t][c]) lives in the v-tile slot OFF_V from its build (under
// the second level pair's GEMM in the fused kernel, under the W/U GEMM in the prep kernel) to C3
// or its store.
// beta K Gamma and beta V (MN-major [t][.], 16 KB each) live in the A1 slot from P3 until
// the W/U GEMM has read them; then A1 takes W^T (and, in the prep kernel, (Q Gamma)^T).
constexpr uint32_t OFF_BKG = OFF_A1, OFF_BV = OFF_A1 + 16384;

struct Misc {
    alignas(16) float beta[C];
    alignas(16) float diag[16][16];
    alignas(16) uint64_t bar_qkz;  // TMA: q, k tiles of a chunk (and its z tile in the prep kernel)
    uint64_t bar_z;                // TMA: z tile of a chunk (fused kernel)
    uint64_t bar_v;                // TMA: v tile of a chunk
    uint64_t bar_m0, bar_m1;       // tensor-core commits, alternating
    uint32_t tmem_base;
    int next_item;                 // fused kernel: the work item taken for after this one
};
static_assert(offsetof(Misc, beta) % 16 == 0 &&
                  offsetof(Misc, bar_qkz) % 8 == 0 && OFF_MISC % 16 == 0,
              "shared-memory block alignment");
constexpr uint32_t SMEM_BYTES = OFF_MISC + sizeof(Misc) + 1024;

// ---- TMEM columns (512 allocated)
constexpr uint32_t TM_S = 0;      // fp32 state, lanes = key channel c, cols = v   (128)
constexpr uint32_t TM_LVL = 384;  // two level-pair score tiles                    (2 x 64)
constexpr uint32_t TM_MG = 384;   // the inverse's merge products                  (2 x 64)
constexpr uint32_t TM_D1 = 256;   // [(W S)^T | (Q Gamma S)^T], + (M Delta)^T above (128)
constexpr uint32_t TM_W = 384;    // W^T                                           (64)
constexpr uint32_t TM_U = 448;    // U^T                                           (64)

constexpr uint32_t IDESC_LVL = tc::idesc_bf16(128, 64, 0, 0);
constexpr uint32_t IDESC_WU = tc::idesc_bf16(128, 64, 1, 0);
constexpr uint32_t IDESC_QU = tc::idesc_bf16(128, 64, 0, 0);
constexpr uint32_t IDESC_SW = tc::idesc_bf16(128, 64, 1, 1);   // C1, W half (B MN-major)
constexpr uint32_t IDESC_SG = tc::idesc_bf16(128, 64, 1, 0);   // C1, Q Gamma half (B K-major)
constexpr uint32_t IDESC_SK = tc::idesc_bf16(128, 128, 1, 0);
constexpr uint32_t IDESC_MG64 = tc::idesc_bf16(128, 64, 0, 1);  // inverse merges
constexpr uint32_t IDESC_MG32 = tc::idesc_bf16(128, 32, 0, 1);

// G2 (fp32, 64 tokens x 128 channels) keeps each row as two halves: channel
// c = 8 a + 4 h + j sits at 64 h + 4 a + j, so that both the 8-channel groups read by
// (token, 8 channels) items and the 4-channel groups read by (token, lane) items are
// contiguous across a warp.
__device__ __forceinline__ int gsw(int c) { return ((c >> 2) & 1) * 64 + (c >> 3) * 4 + (c & 3); }
__device__ __forceinline__ int g4off(int lane) { return (lane & 1) * 64 + (lane >> 1) * 4; }
__device__ __forceinline__ void load8g(const float* G2, int t, int c8, float (&f)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(G2 + t * 128 + c8 * 4);
    const float4 b = *reinterpret_cast<const float4*>(G2 + t * 128 + 64 + c8 * 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
// softplus(x) = max(x, 0) + log(1 + e^{-|x|}) with the hardware exp2/log2 approximations.
__device__ __forceinline__ float softplus_fast(float x) {
    return fmaxf(x, 0.f) + __logf(1.f + __expf(-fabsf(x)));
}

// This thread's two (token, 8-channel) items of the level operands: t = tid/16 + 32 r,
// channels 8 (tid % 16) ..; loaded once per chunk and shared by the four level builds.
struct LevelItems {
    uint4 k[2], q[2];
    float g[2][8];
};

__device__ __forceinline__ void load_level_items(const uint8_t* sm, int tid, LevelItems& it) {
    const float* G2 = reinterpret_cast<const float*>(sm + OFF_G);
    const int c8 = tid & 15;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int t = (tid >> 4) + 32 * r;
        it.k[r] = *reinterpret_cast<const uint4*>(sm + OFF_K + t * 256 + c8 * 16);
        it.q[r] = *reinterpret_cast<const uint4*>(sm + OFF_Q + t * 256 + c8 * 16);
        load8g(G2, t, c8, it.g[r]);
    }
}

// Level li (half-width h = 32 >> li) splits every 2h-block of tokens into a lower and an
// upper half; a token's rank among the 32 tokens of its half is its index with bit log2(h)
// removed.  Two levels share one GEMM: the A operand (128 rows) holds, per level slot
// (li & 1), the upper-half k_t (rows 64 slot + rank) and q_t (rows 64 slot + 32 + rank) scaled
// by e^{G_t - G_r}; the B operand (64 rows) holds the lower-half k_i (rows 32 slot + rank)
// scaled by e^{G_r - G_i}, r the last token of the lower half.  Both factors are <= 1.  The
// product's diagonal 64 x 32 blocks are the two levels' scores; G2 is in log2 units, so every
// factor is one ex2 of a difference <= 0.
__device__ __forceinline__ int level_rank(int t, int s) {
    return ((t >> (s + 1)) << s) | (t & ((1 << s) - 1));
}
__device__ __forceinline__ void build_level(uint8_t* sm, int li, int tid, const LevelItems& it) {
    const float* G2 = reinterpret_cast<const float*>(sm + OFF_G);
    const int c8 = tid & 15;
    const int s = 5 - li, h = 1 << s, slot = li & 1;
    uint8_t* A = sm + OFF_LVL + LV_PA;
    uint8_t* Bop = sm + OFF_LVL + LV_PB;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int t = (tid >> 4) + 32 * r;
        const int ref = (t & ~(2 * h - 1)) + h - 1;
        const bool upper = (t & h) != 0;
        const int rank = level_rank(t, s);
        float r8[8], f[8];
        load8g(G2, ref, c8, r8);
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = ex2(upper ? it.g[r][j] - r8[j] : r8[j] - it.g[r][j]);
        const uint4 kv = scale8_bf16(it.k[r], f);
        if (upper) {
            *reinterpret_cast<uint4*>(A + kmaj_off(64 * slot + rank, c8 * 8, 128)) = kv;
            *reinterpret_cast<uint4*>(A + kmaj_off(64 * slot + 32 + rank, c8 * 8, 128)) =
                scale8_bf16(it.q[r], f);
        } else {
            *reinterpret_cast<uint4*>(Bop + kmaj_off(32 * slot + rank, c8 * 8, 64)) = kv;
        }
    }
}

// Pairs inside the 4-token block b4: the exact pairwise decay e^{G_t - G_i} per channel on
// CUDA cores (one warp, lane = channels 4 lane .. 4 lane + 3), dot products reduced over the
// lanes into ms.diag[b4]: [0, 6) the A pairs, [6, 10) M's diagonal, [10, 16) the M pairs.
__device__ __forceinline__ void diag_block(const uint8_t* sm, Misc& ms, int b4, int lane) {
    const float* G2 = reinterpret_cast<const float*>(sm + OFF_G);
    const int c4 = lane * 4;
    float kk[4][4], qq[4][4], gg[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int t = 4 * b4 + a;
        const uint2 kr = *reinterpret_cast<const uint2*>(sm + OFF_K + t * 256 + c4 * 2);
        const uint2 qr = *reinterpret_cast<const uint2*>(sm + OFF_Q + t * 256 + c4 * 2);
        kk[a][0] = bf_lo(kr.x); kk[a][1] = bf_hi(kr.x); kk[a][2] = bf_lo(kr.y); kk[a][3] = bf_hi(kr.y);
        qq[a][0] = bf_lo(qr.x); qq[a][1] = bf_hi(qr.x); qq[a][2] = bf_lo(qr.y); qq[a][3] = bf_hi(qr.y);
        const float4 g = *reinterpret_cast<const float4*>(G2 + t * KD + g4off(lane));
        gg[a][0] = g.x; gg[a][1] = g.y; gg[a][2] = g.z; gg[a][3] = g.w;
    }
    float v[16];
#pragma unroll
    for (int a = 0; a < 4; ++a) {  // M diagonal
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) s = fmaf(qq[a][j], kk[a][j], s);
        v[6 + a] = s;
    }
    // e^{G_a - G_b} = the product of e^{G_s - G_{s-1}} over b < s <= a: three ex2 per channel
    float ee[4][4];
#pragma unroll
    for (int a = 1; a < 4; ++a)
#pragma unroll
        for (int j = 0; j < 4; ++j) ee[a][j] = ex2(gg[a][j] - gg[a - 1][j]);
#pragma unroll
    for (int a = 1; a < 4; ++a) {
        float dec[4] = {1.f, 1.f, 1.f, 1.f};
#pragma unroll
        for (int b = a - 1; b >= 0; --b) {
            float sa = 0.f, sq = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                dec[j] *= ee[b + 1][j];
                const float kd = kk[b][j] * dec[j];
                sa = fmaf(kk[a][j], kd, sa);
                sq = fmaf(qq[a][j], kd, sq);
            }
            const int idx = a * (a - 1) / 2 + b;
            v[idx] = sa;
            v[10 + idx] = sq;
        }
    }
    // reduce-scatter over the 32 lanes: lane l ends with value (l >> 1) & 15
#pragma unroll
    for (int off = 16, w = 8; off >= 2; off >>= 1, w >>= 1) {
        const bool hi = (lane & off) != 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < w) {
                const float send = hi ? v[j] : v[j + w];
                const float keep = hi ? v[j + w] : v[j];
                v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
        }
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    if ((lane & 1) == 0) ms.diag[b4][lane >> 1] = v[0];
}

// beta K Gamma and beta V as MN-major [t][.] operands in the A1 slot, for the same
// (token, 8 channels) items as the level operands (k and G from their registers).
__device__ __forceinline__ void build_bkg_bv(uint8_t* sm, const Misc& ms, int tid,
                                             const LevelItems& items) {
#pragma unroll
    for (int ii = 0; ii < 2; ++ii) {
        // the same (token, 8 channels) items as the level operands: k and G from registers
        const int item = tid + NT * ii, tt = item >> 4, c8 = item & 15;
        const float bt = ms.beta[tt];  // a bf16 value, so bt * v rounds once, as in fp32
        float f[8], b8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            f[j] = bt * ex2(items.g[ii][j]);
            b8[j] = bt;
        }
        *reinterpret_cast<uint4*>(sm + OFF_BKG + mnmaj_off(tt, c8 * 8, 8192)) = scale8_bf16(items.k[ii], f);
        *reinterpret_cast<uint4*>(sm + OFF_BV + mnmaj_off(tt, c8 * 8, 8192)) =
            scale8_bf16(*reinterpret_cast<const uint4*>(sm + OFF_V + tt * 256 + c8 * 16), b8);
    }
}

// K~ = K e^{G_last - G} as the MN-major [t][c] operand in the v-tile slot, for the same
// (token, 8 channels) items as the level operands (k and G from their registers).
__device__ __forceinline__ void build_kt(uint8_t* sm, int tid, const LevelItems& items) {
    const float* G2 = reinterpret_cast<const float*>(sm + OFF_G);
    const int c8 = tid & 15;
    float gl[8];
    load8g(G2, 63, c8, gl);
#pragma unroll
    for (int ii = 0; ii < 2; ++ii) {
        const int tt = (tid >> 4) + 32 * ii;
        float f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = ex2(gl[j] - items.g[ii][j]);
        *reinterpret_cast<uint4*>(sm + OFF_V + mnmaj_off(tt, c8 * 8, 8192)) = scale8_bf16(items.k[ii], f);
    }
}

// Float index of element (t, i) of a 64 x 64 fp32 matrix whose 16-byte column groups are
// XOR-swizzled by the row, so that row-wise and column-wise float4 accesses by
// consecutive threads fall into distinct banks.
__device__ __forceinline__ int swz(int t, int i) {
    return t * 64 + ((((i >> 2) ^ (t & 15))) << 2) + (i & 3);
}

// What the chunk-parallel prep kernel writes per work item (one chunk of one sequence):
// W^T (MN-major [c][t]) through the tile map tm_wq (z = 2 item), Q Gamma (K-major [t][c], two
// 64-channel atoms) through tm_qg over the same array (z = 4 item + 2, 4 item + 3), U^T through
// tm_uu and K~ through tm_kt (z = item), the M tile (its shared-memory bytes) at
// mm + kItemMM item and Gamma_last (fp32) at gl + 128 item.  Items are the chunks
// [seg_n0, seg_n0 + seg_len) of every sequence, item = bh * seg_len + (n - seg_n0).
struct PrepSeg {
    int seg_n0, seg_len, items;
    uint8_t* mm;
    float* gl;
};

// Work items of the fused kernel: item i is segment j = i / BH (chunks [j seg_len,
// (j + 1) seg_len)) of sequence i % BH.  With `counter` null every CTA takes item blockIdx.x
// (one whole sequence, seg_len = all chunks).  Otherwise a grid of at most one CTA per SM
// takes items from *counter in order; the fp32 state passes from a sequence's segment j - 1
// to segment j through `handoff` (B, H, K, V), and flags[bh] = j says that it is there.
// Items are handed out segment-major, so the item a CTA waits for was taken earlier by a
// CTA that is running: the waits always end.
struct FusedSched {
    int BH, seg_len, n_items;
    int* counter;
    unsigned* flags;
    float* handoff;
};

// The chunk loop shared by the fused kernel (kSplit = false: one CTA per sequence, the
// state carried in TMEM from chunk to chunk) and the prep kernel (kSplit = true: CTAs
// stride over the chunks of all sequences, and everything that does not depend on the
// state is written out for the carry kernel).
template <bool kSplit>
__device__ __forceinline__ void chunk_loop(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                           const CUtensorMap* tm_v, const CUtensorMap* tm_z,
                                           const CUtensorMap* tm_wq, const CUtensorMap* tm_qg,
                                           const CUtensorMap* tm_uu, const CUtensorMap* tm_kt,
                                           int H, int T,
                                           const __nv_bfloat16* __restrict__ beta,
                                           const float* __restrict__ A_log,
                                           const float* __restrict__ dt_bias, float scale,
                                           const float* __restrict__ h0,
                                           __nv_bfloat16* __restrict__ out, float* __restrict__ hT,
                                           PrepSeg seg, FusedSched fs) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    const uint32_t sb = tc::smem_u32(sm);
    Misc& ms = *reinterpret_cast<Misc*>(sm + OFF_MISC);
    float* G2 = reinterpret_cast<float*>(sm + OFF_G);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // TMEM is read in 32-lane quarters: warp w reaches lanes 32*(w & 3) .. +31; the four
    // warps sharing a quarter split the columns by `part`.
    const int q4 = warp & 3, part = warp >> 2, row = q4 * 32 + lane;
    const int nchunks = (T + C - 1) / C;
    // Work items.  Prep kernel: one chunk each, every gridDim.x-th item of the segment.
    // Fused kernel: a segment of one sequence's chunks (see FusedSched).
    const int n_items = kSplit ? seg.items : fs.n_items;
    const bool dynamic = !kSplit && fs.counter != nullptr;
    auto item_bh = [&](int it) -> size_t {
        return kSplit ? (size_t)(it / seg.seg_len) : (size_t)(it % fs.BH);
    };
    auto item_nb = [&](int it) -> int {  // first chunk of the item
        return kSplit ? seg.seg_n0 + it % seg.seg_len : (it / fs.BH) * fs.seg_len;
    };
    auto item_ne = [&](int it) -> int {  // one past its last chunk
        return kSplit ? item_nb(it) + 1 : min(nchunks, item_nb(it) + fs.seg_len);
    };
    for (int i = tid; i < (int)(OFF_MISC / 16); i += NT)
        reinterpret_cast<uint4*>(sm)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
        tc::mbar_init(&ms.bar_qkz, 1);
        tc::mbar_init(&ms.bar_z, 1);
        tc::mbar_init(&ms.bar_v, 1);
        tc::mbar_init(&ms.bar_m0, 1);
        tc::mbar_init(&ms.bar_m1, 1);
        tc::fence_barrier_init();
        if (dynamic) ms.next_item = atomicAdd(fs.counter, 1);
        tc::tma_prefetch_desc(tm_q);
        tc::tma_prefetch_desc(tm_k);
        tc::tma_prefetch_desc(tm_v);
        tc::tma_prefetch_desc(tm_z);
    }
    if (warp == 0) {
        tc::tmem_alloc(&ms.tmem_base, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = ms.tmem_base;

    uint32_t ph_qkz = 0, ph_z = 0, ph_v = 0, ph0 = 0, ph1 = 0;
    bool failed = false;
    const bool group_c = warp < 8;  // fused: carry group; warps 8-15 form the gate group
    // the current chunk: item cur_it, chunk cur_n of its sequence
    int cur_it = dynamic ? ms.next_item : (int)blockIdx.x;
    int cur_n = cur_it < n_items ? item_nb(cur_it) : 0;
    if (tid == 0 && cur_it < n_items) {
        const int bh0 = (int)item_bh(cur_it), y0 = cur_n * C;
        uint64_t* zb = kSplit ? &ms.bar_qkz : &ms.bar_z;
        tc::mbar_arrive_expect_tx(&ms.bar_qkz, (kSplit ? 3u : 2u) * 16384u);
        if (!kSplit) tc::mbar_arrive_expect_tx(zb, 16384u);
        tc::tma_load_3d(sm + OFF_Q, tm_q, 0, y0, bh0, &ms.bar_qkz);
        tc::tma_load_3d(sm + OFF_K, tm_k, 0, y0, bh0, &ms.bar_qkz);
        tc::tma_load_3d(sm + OFF_LVL + LV_Z, tm_z, 0, y0, bh0, zb);
        tc::mbar_arrive_expect_tx(&ms.bar_v, 16384u);
        tc::tma_load_3d(sm + OFF_V, tm_v, 0, y0, bh0, &ms.bar_v);
    }

    // The fused kernel's state of sequence sbh: fp32 in TMEM (lane c = row) and bf16 as the
    // MN-major operand [c][v], this thread's columns [v0b, v0b + nv).  It comes from h0 (a
    // sequence's first segment) or from the handoff of the previous segment (read past L1:
    // another SM wrote it), and leaves to the handoff or to hT.
    // 32 columns per call, every load issued before the first is used (L2 latency once)
    auto state_in32 = [&](size_t sbh, const float* src, int v0b) {
        const int c = row;
        float4 x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            x[j] = src ? __ldcg(reinterpret_cast<const float4*>(src + (sbh * KD + c) * VD + v0b + 4 * j))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float f[16];
            uint32_t r[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 y = x[4 * h + j];
                f[4 * j] = y.x; f[4 * j + 1] = y.y; f[4 * j + 2] = y.z; f[4 * j + 3] = y.w;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(f[j]);
            tc::tmem_st16(taddr(tmem, warp, TM_S + v0b + 16 * h), r);
            store16_mn(sm + OFF_S, c, v0b + 16 * h, 16384, f);
        }
        tc::tmem_st_wait();
    };
    auto state_out32 = [&](size_t sbh, float* dst, int v0b) {
        const int c = row;
        uint32_t d0[16], d1[16];
        tc::tmem_ld16(taddr(tmem, warp, TM_S + v0b), d0);
        tc::tmem_ld16(taddr(tmem, warp, TM_S + v0b + 16), d1);
        tc::tmem_ld_wait();
        float* p = dst + (sbh * KD + c) * VD + v0b;
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
            *reinterpret_cast<float4*>(p + j) =
                make_float4(__uint_as_float(d0[j]), __uint_as_float(d0[j + 1]),
                            __uint_as_float(d0[j + 2]), __uint_as_float(d0[j + 3]));
            *reinterpret_cast<float4*>(p + 16 + j) =
                make_float4(__uint_as_float(d1[j]), __uint_as_float(d1[j + 1]),
                            __uint_as_float(d1[j + 2]), __uint_as_float(d1[j + 3]));
        }
    };
    if (!kSplit && cur_it < n_items) {  // the first item's initial state
        const int j0 = cur_it / fs.BH;
        bool ok = true;
        if (j0 > 0) ok = tid != 0 || tc::flag_wait_geq(fs.flags + item_bh(cur_it), (unsigned)j0);
        if (__syncthreads_or(!ok)) failed = true;
        if (!failed) state_in32(item_bh(cur_it), j0 > 0 ? fs.handoff : h0, 32 * part);
    }

    // Gate of item (gbh, gn) by warps GLO .. GLO + GW - 1 (named barrier 2): waits for its z
    // tile, loads beta, and writes G2 = in-chunk cumulative log2 decay.  The fused kernel runs
    // it on warps 8-15 during the carry; the prep kernel on all warps.
    constexpr int GLO = kSplit ? 0 : 8, GW = kSplit ? 16 : 8, TPW = C / GW;
    // The gate's global reads (beta, dt_bias and A_log of the chunk's head) are issued early
    // by the gate threads, so that their latency is hidden by the tensor-core work in between.
    struct GatePre {  // raw loaded values: nothing here waits for the loads to land
        unsigned short beta_bits;
        float A_log_h;
        float4 dt;
    };
    auto gate_fetch = [&](size_t gbh, int gn) -> GatePre {
        GatePre p;
        // an in-bounds token for every thread; gate_scan keeps the value only for tg < cnn
        const int tg = (warp - GLO) * 32 + lane, tn = gn * C, cnn = min(C, T - tn);
        const int tc = max(0, min(tg, cnn - 1));
        p.beta_bits = __ldg(reinterpret_cast<const unsigned short*>(beta) + gbh * T + tn + tc);
        const int hh = (int)(gbh % H);
        const float* db = dt_bias + (size_t)hh * KD + lane * 4;
        p.dt = make_float4(__ldg(db), __ldg(db + 1), __ldg(db + 2), __ldg(db + 3));
        p.A_log_h = __ldg(A_log + hh);
        return p;
    };
    auto gate_scan = [&](size_t gbh, int gn, const GatePre& gp) -> bool {
        const int wg = warp - GLO;
        const bool ok = !tc::named_sync_or(2, 32 * GW,
                                           !(tid != 32 * GLO ||
                                             tc::mbar_wait(kSplit ? &ms.bar_qkz : &ms.bar_z,
                                                           kSplit ? ph_qkz : ph_z)));
        const int tn = gn * C, cnn = min(C, T - tn);
        const int tg = wg * 32 + lane;
        if (tg < C) ms.beta[tg] = tg < cnn ? __uint_as_float((uint32_t)gp.beta_bits << 16) : 0.f;
        const int c4 = lane * 4;
        const float4 dt = gp.dt;
        const float mult = -expf(gp.A_log_h) * LOG2E;
        // this warp's TPW tokens: running sums in registers; only the warp totals are exchanged
        float4 acc[TPW];
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int a = 0; a < TPW; ++a) {
            const int t = TPW * wg + a;
            const uint2 zr = *reinterpret_cast<const uint2*>(sm + OFF_LVL + LV_Z + t * 256 + c4 * 2);
            const float x0 = bf_lo(zr.x) + dt.x, x1 = bf_hi(zr.x) + dt.y;
            const float x2 = bf_lo(zr.y) + dt.z, x3 = bf_hi(zr.y) + dt.w;
            const float m = (t < cnn) ? mult : 0.f;
            a0 = fmaf(m, softplus_fast(x0), a0);
            a1 = fmaf(m, softplus_fast(x1), a1);
            a2 = fmaf(m, softplus_fast(x2), a2);
            a3 = fmaf(m, softplus_fast(x3), a3);
            acc[a] = make_float4(a0, a1, a2, a3);
        }
        // the warp total goes to the totals slot for the later warps to read (a slot of its
        // own, so the rows below need no second barrier)
        float4* gtot = reinterpret_cast<float4*>(sm + OFF_LVL + (kSplit ? LV_GTP : LV_GTF));
        gtot[wg * 32 + lane] = acc[TPW - 1];
        tc::named_sync(2, 32 * GW);
        float4 pre = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int g = 0; g < wg; ++g) {
            const float4 x = gtot[g * 32 + lane];
            pre.x += x.x; pre.y += x.y; pre.z += x.z; pre.w += x.w;
        }
#pragma unroll
        for (int a = 0; a < TPW; ++a)
            *reinterpret_cast<float4*>(G2 + (TPW * wg + a) * KD + g4off(lane)) =
                make_float4(acc[a].x + pre.x, acc[a].y + pre.y, acc[a].z + pre.z, acc[a].w + pre.w);
        return ok;
    };

    if (cur_it < n_items && (kSplit || !group_c)) {
        const GatePre gp = gate_fetch(item_bh(cur_it), cur_n);
        failed = !gate_scan(item_bh(cur_it), cur_n, gp);
    }
    if constexpr (kSplit) {
        ph_qkz ^= 1u;
        if (__syncthreads_or(failed)) failed = true;
    } else {
        // the first chunk's q and k tiles (the gate waited for its z)
        const bool okq = cur_it >= n_items || tid != 0 || tc::mbar_wait(&ms.bar_qkz, ph_qkz);
        ph_z ^= 1u;
        ph_qkz ^= 1u;
        if (__syncthreads_or(failed || !okq)) failed = true;
    }

// One thread polls the mbarrier; the others sleep in the CTA barrier that follows.
#define KDA_WAIT(bar, ph)                                                \
    do {                                                                 \
        const bool ok_ = tid != 0 || tc::mbar_wait(&ms.bar, ph);         \
        ph ^= 1u;                                                        \
        if (__syncthreads_or(!ok_)) failed = true;                       \
        tc::fence_after_sync();                                          \
    } while (0)
#define KDA_SYNC_FOR_MMA()                                               \
    do {                                                                 \
        tc::fence_proxy_async_smem();                                    \
        tc::fence_before_sync();                                         \
        __syncthreads();                                                 \
        tc::fence_after_sync();                                          \
    } while (0)
// The GEMM of one level pair (operands built by build_level), committed to `bar`.
#define KDA_PAIR_MMA(col, bar)                                           \
    do {                                                                 \
        if (tid == 0) {                                                  \
            _Pragma("unroll") for (int ks = 0; ks < 8; ++ks)             \
                tc::mma_bf16(tmem + (col), desc_k(sb + OFF_LVL + LV_PA, 128, ks), \
                             desc_k(sb + OFF_LVL + LV_PB, 64, ks), IDESC_LVL, ks > 0); \
            tc::mma_commit(&ms.bar);                                     \
        }                                                                \
    } while (0)

    // The output of a chunk, o = scale (Q Gamma S + M Delta) from TMEM (lanes = v), is written
    // during the next chunk's inverse, by warps that the forward substitution leaves idle, or
    // after the loop for the last chunk: (o_bh, o_t0, o_cn) name the chunk whose o is pending.
    bool o_pend = false, s_pend = false;
    size_t o_bh = 0;
    int o_t0 = 0, o_cn = 0;
    // The previous chunk's output, this warp's lanes (columns v = row) and tokens [tb0, tb0 + ntb):
    // straight to global memory, or (staged) into the free state-copy slot as a bf16 [t][v] tile
    // that one bulk copy then writes (o_store).
    auto o_emit = [&](int tb0, int ntb, bool staged) {
#pragma unroll 1
        for (int tb = tb0; tb < tb0 + ntb; tb += 16) {
            uint32_t dq[16];
            tc::tmem_ld16(taddr(tmem, warp, TM_D1 + 64 + tb), dq);
            tc::tmem_ld_wait();
            float o[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = scale * __uint_as_float(dq[j]);
            if (staged) {
                __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(sm + OFF_S) + tb * VD + row;
#pragma unroll
                for (int j = 0; j < 16; ++j) st[j * VD] = __float2bfloat16_rn(o[j]);
            } else {
                store_o16_pairs(out + (o_bh * T + o_t0 + tb) * VD, row, lane, o_cn - tb, o);
            }
        }
    };
    // The staged output tile (rows below o_cn) to global memory, by thread 0 after a barrier.
    auto o_store = [&]() {
        tc::bulk_store(out + (o_bh * T + o_t0) * VD, sm + OFF_S, (uint32_t)(o_cn * VD * 2));
        tc::bulk_commit();
    };
    while (cur_it < n_items && !failed) {
        const int it = cur_it;
        const size_t bh = item_bh(it);
        const int t0 = cur_n * C, cn = min(C, T - t0);
        const int seg_j = kSplit ? 0 : it / fs.BH;
        const bool last_of_item = cur_n + 1 >= item_ne(it);
        // The chunk after this one: the next of this item, or the first of the next item.  A
        // dynamic fused kernel takes that item now; it is known to all threads after the
        // first barrier below (next_pending).
        int nxt_it = last_of_item ? (kSplit ? it + (int)gridDim.x : n_items) : it;
        const bool next_pending = dynamic && last_of_item;
        if (next_pending && tid == 0) ms.next_item = atomicAdd(fs.counter, 1);
        bool has_next = !next_pending && nxt_it < n_items;
        size_t nbh = has_next ? item_bh(nxt_it) : bh;
        int nt0 = has_next ? (last_of_item ? item_nb(nxt_it) : cur_n + 1) * C : t0;
        // ---------------------------------------------------------------- P3: levels 32, 16
        // one GEMM per pair of levels; the first pair's runs under the next phase
        LevelItems items;
        load_level_items(sm, tid, items);
        build_level(sm, 0, tid, items);
        build_level(sm, 1, tid, items);
        KDA_SYNC_FOR_MMA();
        KDA_PAIR_MMA(TM_LVL, bar_m0);
        if (next_pending) {
            nxt_it = ms.next_item;
            has_next = nxt_it < n_items;
            nbh = has_next ? item_bh(nxt_it) : bh;
            nt0 = has_next ? item_nb(nxt_it) * C : t0;
        }
        // ---------------------------------------------------------------- P3: 4-token blocks
        // under the first pair's GEMM: the 4-token blocks (prep kernel; the fused kernel's gate
        // group did them during the previous carry) or beta K Gamma / beta V (fused kernel)
        bool okv_all = true;
        if constexpr (kSplit) {
            diag_block(sm, ms, warp, lane);
        } else {
            okv_all = tc::mbar_wait(&ms.bar_v, ph_v);
            build_bkg_bv(sm, ms, tid, items);
        }
        {
            const bool okv = kSplit ? (tid != 0 || tc::mbar_wait(&ms.bar_v, ph_v)) : okv_all;
            const bool ok0 = tid != 0 || tc::mbar_wait(&ms.bar_m0, ph0);
            ph_v ^= 1u; ph0 ^= 1u;
            if (__syncthreads_or(!(okv && ok0))) failed = true;
            tc::fence_after_sync();
            if (failed) break;
        }
        // ---------------------------------------------------------------- P3: levels 8, 4
        build_level(sm, 2, tid, items);
        build_level(sm, 3, tid, items);
        KDA_SYNC_FOR_MMA();
        KDA_PAIR_MMA(TM_LVL + 64, bar_m1);
        // while the second pair's GEMM runs: beta K Gamma and beta V (prep kernel), or K~ =
        // K e^{G_last - G} from the level items' registers into the v slot, whose v tile the
        // beta V build has already consumed, and the pairs inside 4-token blocks (fused kernel)
        if constexpr (kSplit) {
            build_bkg_bv(sm, ms, tid, items);
        } else {
            build_kt(sm, tid, items);
            diag_block(sm, ms, warp, lane);  // the pairs inside 4-token blocks, one block per warp
        }
        KDA_WAIT(bar_m1, ph1);
        if (failed) break;
        // ---------------------------------------------------------------- P3 epilogue
        {
            float* Af = reinterpret_cast<float*>(sm + OFF_LVL + LV_AF);
            uint8_t* MB = sm + OFF_LVL + LV_MB;
            // (a) level scores.  TMEM lane `row` of the tile of pair part / 2: rows 64 slot ..
            //     belong to level li = 2 (part / 2) + slot, k rows (A scores) first, then q rows
            //     (M scores), by the upper token's rank; the level's 32 columns are the lower
            //     tokens' ranks.  Only pairs inside one 2h-block are scores.
            {
                const int p = part >> 1, slot = row >> 6, s = 5 - (2 * p + slot), h = 1 << s;
                const bool is_m = (row & 32) != 0;
                const int rt = row & 31, rb = 16 * (part & 1);
                const int t = ((rt >> s) << (s + 1)) | h | (rt & (h - 1));
                uint32_t d[16];
                tc::tmem_ld16(taddr(tmem, warp, TM_LVL + 64 * p + 32 * slot + rb), d);
                tc::tmem_ld_wait();
                // The valid columns of this thread's 16 form one run of len = min(h, 16) starting at
                // a multiple of len (none when the run lies in the other 16): move it to the front
                // with selects, so the stores below index registers statically.
                const int blk = rt >> s, len = min(h, 16);
                const int j0 = (blk << s) - rb;  // first valid column; the run is [j0, j0 + len)
                const bool any = j0 < 16 && j0 + h > 0;
                const int i0 = rb + max(j0, 0) + (blk << s);  // token of the run's first column
                float w[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) w[k] = __uint_as_float(d[k]);
                if (len <= 8) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) w[k] = (j0 & 8) ? w[8 + k] : w[k];
                }
                if (len <= 4) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) w[k] = (j0 & 4) ? w[4 + k] : w[k];
                }
                // the run is 4, 8 or 16 consecutive tokens from i0 (a multiple of its length):
                // whole 8- or 16-byte stores
                if (any && is_m) {
                    uint32_t pk[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m) pk[m] = tc::pack_bf16x2(w[2 * m], w[2 * m + 1]);
                    if (len == 4) {
                        *reinterpret_cast<uint2*>(MB + kmaj_off(t, i0, 64)) = make_uint2(pk[0], pk[1]);
                    } else {
                        *reinterpret_cast<uint4*>(MB + kmaj_off(t, i0, 64)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        if (len == 16)
                            *reinterpret_cast<uint4*>(MB + kmaj_off(t, i0 + 8, 64)) =
                                make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                } else if (any && p == 0) {
                    // levels 32 and 16 lie off the 16 x 16 diagonal blocks: bf16, for the merges
                    const float bt = ms.beta[t];
                    float a16[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) a16[k] = bt * w[k];
                    store16_k(sm + OFF_LVL + LV_AB, t, i0, 64, a16);
                } else if (any) {
                    const float bt = ms.beta[t];
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        if (4 * m < len)
                            *reinterpret_cast<float4*>(Af + swz(t, i0 + 4 * m)) =
                                make_float4(bt * w[4 * m], bt * w[4 * m + 1], bt * w[4 * m + 2], bt * w[4 * m + 3]);
                }
            }
            // (b) row t, 4-column groups 2 g8, 2 g8 + 1: the 4-token block on the diagonal from the
            //     CUDA-core dot products (A strictly below the diagonal, M on and below), M zero
            //     above it.  A above the diagonal is never read.
            {
                const int t = tid >> 3, g8 = tid & 7, tb = t >> 2, tl = t & 3;
                const float* dg = ms.diag[tb];
                const float bt = ms.beta[t];
#pragma unroll
                for (int hg = 0; hg < 2; ++hg) {
                    const int g = 2 * g8 + hg;
                    if (g < tb) continue;  // level scores, written in (a)
                    float m4[4] = {0.f, 0.f, 0.f, 0.f};
                    if (g == tb) {
                        float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int il = 0; il < 4; ++il) {
                            if (il < tl) {
                                a4[il] = bt * dg[((tl * (tl - 1)) >> 1) + il];
                                m4[il] = dg[10 + ((tl * (tl - 1)) >> 1) + il];
                            } else if (il == tl) {
                                m4[il] = dg[6 + tl];
                            }
                        }
                        *reinterpret_cast<float4*>(Af + swz(t, 4 * g)) = make_float4(a4[0], a4[1], a4[2], a4[3]);
                    }
                    *reinterpret_cast<uint2*>(MB + kmaj_off(t, 4 * g, 64)) =
                        make_uint2(tc::pack_bf16x2(m4[0], m4[1]), tc::pack_bf16x2(m4[2], m4[3]));
                }
            }
        }
        tc::fence_before_sync();
        __syncthreads();
        bool mok = true;  // this thread's waits for the inverse's merge products
        // ---------------------------------------------------------------- P4: T = (I + A)^{-1}
        // T (bf16, K-major [t][i] in LV_TB) blockwise: the four 16 x 16 diagonal blocks by
        // forward substitution on CUDA cores in fp32 (from the diagonal blocks of Af), then the
        // block merges T_RC = -T_RR A_RC T_CC as tcgen05 products (bf16 operands, fp32
        // accumulation): 16 -> 32 for both halves at once, then 32 -> 64.
        {
            const float* Af = reinterpret_cast<const float*>(sm + OFF_LVL + LV_AF);
            uint8_t* TB = sm + OFF_LVL + LV_TB;
            // (a) the diagonal blocks, one column each (left-looking: x_t = delta_tj -
            //     sum_{i<t} A_ti x_i); the other threads clear the off-diagonal blocks of T
            //     and the blocks of A_bf that the merges multiply by zero.
            if (tid < 64) {
                const int R = tid >> 4, j = tid & 15;
                const float* Ab = Af + 16 * R * 64;  // rows 16R.. ; (row & 15) == t
                float x[16];
                // the strictly lower part of this block row by row, in 16-byte groups, each
                // row's loads issued two rows ahead of its use (three rows in registers)
                float4 ar[3][4];
                auto load_row = [&](int t) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (4 * q < t)
                            ar[t % 3][q] = *reinterpret_cast<const float4*>(Ab + t * 64 + (((4 * R + q) ^ t) << 2));
                };
                load_row(1);
                load_row(2);
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    if (t >= 1 && t + 2 < 16) load_row(t + 2);
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (4 * q < t) {
                            const float4 aq = ar[t % 3][q];
                            const float av[4] = {aq.x, aq.y, aq.z, aq.w};
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                if (4 * q + u < t) acc[u] = fmaf(av[u], x[4 * q + u], acc[u]);
                        }
                    }
                    x[t] = ((t == j) ? 1.f : 0.f) - ((acc[0] + acc[1]) + (acc[2] + acc[3]));
                }
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    *reinterpret_cast<__nv_bfloat16*>(TB + kmaj_off(16 * R + t, 16 * R + j, 64)) =
                        __float2bfloat16_rn(x[t]);
                // then the previous chunk's output, tokens 0..15 of this warp's lane quarter
                if (!kSplit && o_pend) o_emit(0, 16, s_pend);
            } else {
                // 16-byte groups of zeros: the 12 off-diagonal 16 x 16 blocks of T, and the 10
                // blocks of A_bf on or above the diagonal (the merges read them against zeros
                // of T; they must hold finite values)
                for (int e = tid - 64; e < 22 * 32; e += NT - 64) {
                    const int blk = e >> 5, q = e & 31;
                    int R, Cb;
                    uint8_t* base;
                    if (blk < 12) {
                        R = blk / 3;
                        Cb = blk % 3 + (blk % 3 >= R ? 1 : 0);
                        base = TB;
                    } else {
                        const int b2 = blk - 12;  // (R, Cb >= R) in row order
                        R = b2 < 4 ? 0 : (b2 < 7 ? 1 : (b2 < 9 ? 2 : 3));
                        Cb = R + b2 - (R == 0 ? 0 : (R == 1 ? 4 : (R == 2 ? 7 : 9)));
                        base = sm + OFF_LVL + LV_AB;
                    }
                    *reinterpret_cast<uint4*>(base + kmaj_off(16 * R + (q >> 1), 16 * Cb + 8 * (q & 1), 64)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                // the previous chunk's output (fused kernel): 16 tokens per warp, 16 (warp / 4)
                // .. of its TMEM lane quarter (warps 0 and 1 take tokens 0..15 of theirs after
                // the substitution).  Staged in the state-copy slot unless that holds this
                // chunk's state already (an item change loaded it: s_pend false).
                if (!kSplit && o_pend) {
                    const int j = warp >> 2;
                    o_emit(16 * j, 16, s_pend);
                }
            }
            const bool o_staged = !kSplit && o_pend && s_pend;
            o_pend = false;
            KDA_SYNC_FOR_MMA();
            if (o_staged && tid == 0) o_store();
            // The four merge products.  Each is M = 128 rows of which the first 64 (or 32) are
            // the blocks' rows: the other rows read whatever follows in shared memory and their
            // results are never read.  T (LV_TB) serves as the K-major A operand [t][i] and, read
            // MN-major, as the B operand T[k][n]; products go back to shared memory in the same
            // K-major layout (row = TMEM lane) and are read MN-major by the next product.
            // (b) 16 -> 32, first product: P = A_bf T_d  (T_d = the diagonal blocks; blocks (1,0)
            //     and (3,2) of P are A_10 T_00 and A_32 T_22)
            // Only the warps that read a product back wait for it (each thread on the mbarrier
            // itself), and they hand the tiles they write to the issuing thread 0 (warp 0)
            // through named barriers among themselves; the other warps go on to the barrier
            // before P5.  A timed-out wait skips its tile and is counted at that barrier.  A
            // warp that waits on an mbarrier waits for every phase of it in turn (a parity
            // wait cannot tell a phase from the one two before it).
            const bool w_b = q4 < 2;                                        // warps 0,1,4,5,8,9,12,13
            const bool w_c = (q4 == 0 && part == 0) || (q4 == 1 && part == 2);  // warps 0, 9
            const bool w_d = q4 == 1 && part < 2;                           // warps 1, 5
            const bool w_e = q4 == 0 && part < 2;                           // warps 0, 4
            if (tid == 0) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + TM_MG, desc_k(sb + OFF_LVL + LV_AB, 64, ks),
                                 desc_mn(sb + OFF_LVL + LV_TB, 8192, ks), IDESC_MG64, ks > 0);
                tc::mma_commit(&ms.bar_m0);
            }
            if (w_b) {  // rows 0..63 of P -> bf16 tile LV_MG
                mok = tc::mbar_wait(&ms.bar_m0, ph0);
                tc::fence_after_sync();
                if (mok) {
                    uint32_t d[16];
                    tc::tmem_ld16(taddr(tmem, warp, TM_MG + 16 * part), d);
                    tc::tmem_ld_wait();
                    float f[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(d[j]);
                    store16_k(sm + OFF_LVL + LV_MG, row, 16 * part, 64, f);
                }
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                tc::named_sync(3, 256);
            }
            ph0 ^= 1u;
            // (c) second product: Q = T_d P;  T_10 = -Q[16:32, 0:16], T_32 = -Q[48:64, 32:48]
            if (tid == 0 && mok) {
                tc::fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + TM_MG + 64, desc_k(sb + OFF_LVL + LV_TB, 64, ks),
                                 desc_mn(sb + OFF_LVL + LV_MG, 8192, ks), IDESC_MG64, ks > 0);
                tc::mma_commit(&ms.bar_m1);
            }
            if (w_c || w_e) {
                // (warp 4 waits here too although it reads nothing of this product: a parity
                // wait must not skip a phase, and warp 4 waits for the next one in (e))
                mok = tc::mbar_wait(&ms.bar_m1, ph1) && mok;
                tc::fence_after_sync();
            }
            if (w_c) {
                if (mok) {
                    uint32_t d[16];
                    tc::tmem_ld16(taddr(tmem, warp, TM_MG + 64 + 16 * part), d);
                    tc::tmem_ld_wait();
                    if (lane >= 16) {
                        float f[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) f[j] = -__uint_as_float(d[j]);
                        store16_k(TB, row, 16 * part, 64, f);
                    }
                }
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                tc::named_sync(4, 64);
            }
            ph1 ^= 1u;
            // (d) 32 -> 64, first product: P' = A_bf[:, 0:32] T[0:32, 0:32]; rows 32..63 are
            //     A_21 T_11 (the rest of T's first 32 columns below row 31 is still zero)
            if (tid == 0 && mok) {
                tc::fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    tc::mma_bf16(tmem + TM_MG, desc_k(sb + OFF_LVL + LV_AB, 64, ks),
                                 desc_mn(sb + OFF_LVL + LV_TB, 8192, ks), IDESC_MG32, ks > 0);
                tc::mma_commit(&ms.bar_m0);
            }
            if (w_d) {  // rows 32..63 of P' -> tile rows 0..31
                mok = tc::mbar_wait(&ms.bar_m0, ph0) && mok;
                tc::fence_after_sync();
                if (mok) {
                    uint32_t d[16];
                    tc::tmem_ld16(taddr(tmem, warp, TM_MG + 16 * part), d);
                    tc::tmem_ld_wait();
                    float f[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(d[j]);
                    store16_k(sm + OFF_LVL + LV_MG, lane, 16 * part, 64, f);
                }
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
            }
            if (w_d || warp == 0) tc::named_sync(5, 96);  // warps 1 and 5 to warp 0
            ph0 ^= 1u;
            // (e) second product: Y = T_22 P'[32:64, :] (A from row 32 of T, K = columns 32..63);
            //     T_21 = -Y
            if (tid == 0 && mok) {
                tc::fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    tc::mma_bf16(tmem + TM_MG + 64, desc_k(sb + OFF_LVL + LV_TB + 4096, 64, 2 + ks),
                                 desc_mn(sb + OFF_LVL + LV_MG, 8192, ks), IDESC_MG32, ks > 0);
                tc::mma_commit(&ms.bar_m1);
            }
            if (w_e) {
                mok = tc::mbar_wait(&ms.bar_m1, ph1) && mok;
                tc::fence_after_sync();
                // fused kernel: the z slot is free (A_bf and the merge tiles are read): the next
                // chunk's z tile, for its gate beside this chunk's carry
                if (!kSplit && tid == 0 && has_next && mok) {
                    tc::mbar_arrive_expect_tx(&ms.bar_z, 16384u);
                    tc::tma_load_3d(sm + OFF_LVL + LV_Z, tm_z, 0, nt0, (int)nbh, &ms.bar_z);
                }
                if (mok) {
                    uint32_t d[16];
                    tc::tmem_ld16(taddr(tmem, warp, TM_MG + 64 + 16 * part), d);
                    tc::tmem_ld_wait();
                    float f[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) f[j] = -__uint_as_float(d[j]);
                    store16_k(TB, 32 + lane, 16 * part, 64, f);
                }
            }
            ph1 ^= 1u;
            // the warps that read no merge product back: Q Gamma (bf16, K-major [t][c] in the
            // A slot, which the substitution is done with) for the C1 operand (fused kernel) or
            // the carry kernel's (prep kernel), four (token, 8 channels) items per thread
            if (q4 >= 2) {
                const int i0 = ((warp >> 2) * 2 + (q4 - 2)) * 32 + lane;  // 0..255 over these 8 warps
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int item = i0 + 256 * m, t = item >> 4, c8 = item & 15;
                    float g8[8], qf[8], f[8];
                    load8g(G2, t, c8, g8);
                    unpack8(*reinterpret_cast<const uint4*>(sm + OFF_Q + t * 256 + c8 * 16), qf);
#pragma unroll
                    for (int j = 0; j < 8; ++j) f[j] = qf[j] * ex2(g8[j]);
                    *reinterpret_cast<uint4*>(sm + OFF_LVL + LV_QG + kmaj_off(t, c8 * 8, 64)) = pack8(f);
                }
            }
        }
        // the staged output has left the state-copy slot that this chunk's copy refills next
        if (!kSplit && tid == 0) tc::bulk_wait_read_all();
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        if (__syncthreads_or(!mok)) failed = true;
        tc::fence_after_sync();
        if (failed) break;
        // (fused kernel) q and k are read: request the next chunk's q and k tiles
        if (!kSplit && tid == 0 && has_next) {
            tc::mbar_arrive_expect_tx(&ms.bar_qkz, 2u * 16384u);
            tc::tma_load_3d(sm + OFF_Q, tm_q, 0, nt0, (int)nbh, &ms.bar_qkz);
            tc::tma_load_3d(sm + OFF_K, tm_k, 0, nt0, (int)nbh, &ms.bar_qkz);
        }
        // ---------------------------------------------------------------- P5: W^T, U^T
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t b = desc_k(sb + OFF_LVL + LV_TB, 64, ks);
                tc::mma_bf16(tmem + TM_W, desc_mn(sb + OFF_BKG, 8192, ks), b, IDESC_WU, ks > 0);
                tc::mma_bf16(tmem + TM_U, desc_mn(sb + OFF_BV, 8192, ks), b, IDESC_WU, ks > 0);
            }
            tc::mma_commit(&ms.bar_m0);
        }
        if constexpr (!kSplit) {
            // (fused kernel) the state the previous chunk's C3 left in TMEM: this chunk's bf16
            // operand [c][v] for C1 (unless an item change already loaded it), then
            // S <- diag(Gamma_last) S in place for C3 (the bf16 copy stays unscaled)
            const int c = row, v0 = 32 * part;
            uint32_t d0[16], d1[16];
            tc::tmem_ld16(taddr(tmem, warp, TM_S + v0), d0);
            tc::tmem_ld16(taddr(tmem, warp, TM_S + v0 + 16), d1);
            tc::tmem_ld_wait();
            if (s_pend) {
                float f[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(d0[j]);
                store16_mn(sm + OFF_S, c, v0, 16384, f);
#pragma unroll
                for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(d1[j]);
                store16_mn(sm + OFF_S, c, v0 + 16, 16384, f);
            }
            const float gl = ex2(G2[63 * KD + gsw(c)]);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                d0[j] = __float_as_uint(__uint_as_float(d0[j]) * gl);
                d1[j] = __float_as_uint(__uint_as_float(d1[j]) * gl);
            }
            tc::tmem_st16(taddr(tmem, warp, TM_S + v0), d0);
            tc::tmem_st16(taddr(tmem, warp, TM_S + v0 + 16), d1);
            tc::tmem_st_wait();
            tc::fence_proxy_async_smem();  // the copy is read by C1's first half after the wait
            s_pend = false;
        }
        // and, in the prep kernel, K~ = K e^{G_last - G} -> the v-tile slot (MN-major [t][c])
        if constexpr (kSplit) {
#pragma unroll
            for (int ii = 0; ii < 2; ++ii) {
                const int item = tid + NT * ii, t = item >> 4, c8 = item & 15;
                float g8[8], gl[8], f[8];
                load8g(G2, t, c8, g8);
                load8g(G2, 63, c8, gl);
#pragma unroll
                for (int j = 0; j < 8; ++j) f[j] = ex2(gl[j] - g8[j]);
                *reinterpret_cast<uint4*>(sm + OFF_V + mnmaj_off(t, c8 * 8, 8192)) =
                    scale8_bf16(*reinterpret_cast<const uint4*>(sm + OFF_K + t * 256 + c8 * 16), f);
            }
        }
        KDA_WAIT(bar_m0, ph0);
        if (failed) break;
        // (fused kernel) the state's bf16 copy and Q Gamma are in place: the Q Gamma half of C1
        // now, under the W^T extraction (the carry window's C1 commit covers it; the previous
        // chunk's output has left those TMEM columns during the substitution)
        if (!kSplit && tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_bf16(tmem + TM_D1 + 64, desc_mn(sb + OFF_S, 16384, ks),
                             desc_k(sb + OFF_LVL + LV_QG, 64, ks), IDESC_SG, ks > 0);
        }
        // prep kernel: q and k are free: request the next chunk's q, k and z (on one barrier)
        if (kSplit && tid == 0 && has_next) {
            tc::mbar_arrive_expect_tx(&ms.bar_qkz, 3u * 16384u);
            tc::tma_load_3d(sm + OFF_Q, tm_q, 0, nt0, (int)nbh, &ms.bar_qkz);
            tc::tma_load_3d(sm + OFF_K, tm_k, 0, nt0, (int)nbh, &ms.bar_qkz);
            tc::tma_load_3d(sm + OFF_LVL + LV_Z, tm_z, 0, nt0, (int)nbh, &ms.bar_qkz);
        }
        if constexpr (!kSplit) {
            // (fused kernel) every part: W^T row c, columns 16 part .. -> A1 (U stays in TMEM
            // for the carry, Q Gamma is in the A slot already)
            const int c = row, tb = 16 * part;
            uint32_t d[16];
            tc::tmem_ld16(taddr(tmem, warp, TM_W + tb), d);
            tc::tmem_ld_wait();
            float f[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(d[j]);
            store16_mn(sm + OFF_A1, c, tb, 16384, f);
        } else {
            // (prep kernel) parts 0-1: W^T row c, columns 32*part.. -> A1; parts 2-3: U^T row v
            // -> K-major, in the state-copy slot (which this kernel has free: Q Gamma is in the
            // A slot, where U^T used to go)
            const bool is_u = part >= 2;
            const int cb = 32 * (part & 1);
            const uint32_t col = is_u ? TM_U : TM_W;
            {
                uint32_t d0[16], d1[16];
                tc::tmem_ld16(taddr(tmem, warp, col + cb), d0);
                tc::tmem_ld16(taddr(tmem, warp, col + cb + 16), d1);
                tc::tmem_ld_wait();
                float f0[16], f1[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) { f0[j] = __uint_as_float(d0[j]); f1[j] = __uint_as_float(d1[j]); }
                if (!is_u) {
                    store16_mn(sm + OFF_A1, row, cb, 16384, f0);
                    store16_mn(sm + OFF_A1, row, cb + 16, 16384, f1);
                } else {
                    store16_k(sm + OFF_S, row, cb, 128, f0);
                    store16_k(sm + OFF_S, row, cb + 16, 128, f1);
                }
            }
            if (kSplit && part == 0) seg.gl[(size_t)it * KD + row] = ex2(G2[63 * KD + gsw(row)]);
        }
        KDA_SYNC_FOR_MMA();
        // (without a next item this fetches the current one again, unused)
        const GatePre gp = gate_fetch(nbh, nt0 / C);
        // ---------------------------------------------------------------- S: operands out | next gate
        if (kSplit && tid == 0) {
            // W^T, Q Gamma, U^T, K~ and M are final: out while every warp computes the next
            // item's gate
            tc::tma_store_3d(tm_wq, sm + OFF_A1, 0, 0, 2 * it);
            tc::tma_store_3d(tm_qg, sm + OFF_LVL + LV_QG, 0, 0, 4 * it + 2);
            tc::tma_store_3d(tm_qg, sm + OFF_LVL + LV_QG + 8192, 0, 0, 4 * it + 3);
            tc::tma_store_3d(tm_uu, sm + OFF_S, 0, 0, it);
            tc::tma_store_3d(tm_kt, sm + OFF_V, 0, 0, it);
            tc::tma_store_3d(tm_kt, sm + OFF_V + 8192, 64, 0, it);
            tc::bulk_store(seg.mm + (size_t)it * kItemMM, sm + OFF_LVL + LV_MB, (uint32_t)kItemMM);
            tc::bulk_commit();
        }
        if constexpr (kSplit) {
        // ---------------------------------------------------------------- S2: next gate
            if (has_next && !gate_scan(nbh, nt0 / C, gp)) failed = true;
        // ---------------------------------------------------------------- S3: drain stores
            if (tid == 0) {
                // the stores have read the v-tile slot, A1, Q Gamma, U^T and M: refill / reuse them
                tc::bulk_wait_read_all();
                if (has_next) {
                    tc::mbar_arrive_expect_tx(&ms.bar_v, 16384u);
                    tc::tma_load_3d(sm + OFF_V, tm_v, 0, nt0, (int)nbh, &ms.bar_v);
                }
            }
        } else {
        // ---------------------------------------------------------------- C: carry | next gate
            if (group_c) {
                // C1: D[v][t'] = sum_c S[c][v] W^T[c][t'] (t' < 64), sum_c S[c][v] QG[t'][c]
                //     above; two MMAs of N = 64 per K step, the second with a K-major B
                if (tid == 0) {
    #pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_bf16(tmem + TM_D1, desc_mn(sb + OFF_S, 16384, ks),
                                     desc_mn(sb + OFF_A1, 16384, ks), IDESC_SW, ks > 0);
                    tc::mma_commit(&ms.bar_m0);  // (the Q Gamma half went out after the W/U GEMM)
                }
                {
                    const bool ok = tid != 0 || tc::mbar_wait(&ms.bar_m0, ph0);
                    if (tc::named_sync_or(1, 256, !ok)) failed = true;
                    tc::fence_after_sync();
                }
                // C2: lane v, tokens 32*half..: Delta^T = U^T - (W S)^T -> K-major [v][t] (C3
                //     waits for it)
                const int half = warp >> 2, v = row;
                if (!failed) {
#pragma unroll 1
                    for (int tb = 32 * half; tb < 32 * half + 32; tb += 16) {
                        uint32_t dw[16], du[16];
                        tc::tmem_ld16(taddr(tmem, warp, TM_D1 + tb), dw);
                        tc::tmem_ld16(taddr(tmem, warp, TM_U + tb), du);
                        tc::tmem_ld_wait();
                        float f[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(du[j]) - __uint_as_float(dw[j]);
                        store16_k(sm + OFF_LVL + LV_DELTA, v, tb, 128, f);
                    }
                }
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                tc::named_sync(1, 256);
                tc::fence_after_sync();
                // C3: S += K~^T Delta (K~ in the v-tile slot), and (M Delta)^T onto (QG S)^T:
                //     o = scale (QG S + M Delta) (= scale (Q' S + U') with Q' = QG - M W,
                //     U' = M U) is written during the next chunk's inverse (o_emit): its TMEM
                //     columns live on
                if (tid == 0 && !failed) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_bf16(tmem + TM_S, desc_mn(sb + OFF_V, 8192, ks),
                                     desc_k(sb + OFF_LVL + LV_DELTA, 128, ks), IDESC_SK, 1u);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_bf16(tmem + TM_D1 + 64, desc_k(sb + OFF_LVL + LV_DELTA, 128, ks),
                                     desc_k(sb + OFF_LVL + LV_MB, 64, ks), IDESC_QU, 1u);
                    tc::mma_commit(&ms.bar_m1);
                }
                {
                    const bool ok = failed || tid != 0 || tc::mbar_wait(&ms.bar_m1, ph1);
                    if (tc::named_sync_or(1, 256, !ok)) failed = true;
                    tc::fence_after_sync();
                }
                // K~ is consumed: request the next chunk's v tile into its slot.  The new state's
                // bf16 copy for the next C1 is made under the next chunk's W/U GEMM (s_pend).
                if (tid == 0 && has_next && !failed) {
                    tc::mbar_arrive_expect_tx(&ms.bar_v, 16384u);
                    tc::tma_load_3d(sm + OFF_V, tm_v, 0, nt0, (int)nbh, &ms.bar_v);
                }
                // last chunk of an item (while the gate group finishes the next gate): the state
                // goes to the next segment (handoff, then its flag) or to hT, and the next item's
                // state comes in, unless that item is this one's next segment (already here)
                if (!failed && last_of_item) {
                    const bool more = item_ne(it) < nchunks;
                    float* dst = more ? fs.handoff : hT;
                    if (dst) {
                        state_out32(bh, dst, 64 * half);
                        state_out32(bh, dst, 64 * half + 32);
                    }
                    if (more) __threadfence();
                    tc::fence_before_sync();
                    tc::named_sync(1, 256);
                    tc::fence_after_sync();
                    if (more && tid == 0) tc::st_release_gpu(fs.flags + bh, (unsigned)(seg_j + 1));
                    if (has_next && nxt_it != it + fs.BH) {
                        const int nj = nxt_it / fs.BH;
                        bool ok = true;
                        if (nj > 0) ok = tid != 0 || tc::flag_wait_geq(fs.flags + nbh, (unsigned)nj);
                        if (tc::named_sync_or(1, 256, !ok)) failed = true;
                        if (!failed) {
                            state_in32(nbh, nj > 0 ? fs.handoff : h0, 64 * half);
                            state_in32(nbh, nj > 0 ? fs.handoff : h0, 64 * half + 32);
                        }
                    }
                }
            } else if (has_next) {
                // the next chunk's gate, then the wait for its q and k tiles
                if (!gate_scan(nbh, nt0 / C, gp)) failed = true;
                if (tc::named_sync_or(2, 256, !(tid != 256 || tc::mbar_wait(&ms.bar_qkz, ph_qkz))))
                    failed = true;
            }
            ph0 ^= 1u;  // C1's and C3's commits, waited by the carry group only
            ph1 ^= 1u;
            s_pend = !(last_of_item && has_next && nxt_it != it + fs.BH);
            o_pend = true;  // this chunk's output goes out during the next chunk, or after the loop
            o_bh = bh;
            o_t0 = t0;
            o_cn = cn;
        }
        if (has_next) {
            ph_qkz ^= 1u;
            ph_z ^= 1u;
        }
        // (no proxy fence here: what the async proxy reads next, the threads that write it
        // fence before the barrier that precedes that read)
        tc::fence_before_sync();
        if (__syncthreads_or(failed)) failed = true;
        tc::fence_after_sync();
        if (last_of_item) {
            cur_it = nxt_it;
            cur_n = has_next ? item_nb(nxt_it) : 0;
        } else {
            ++cur_n;
        }
    }
#undef KDA_WAIT
#undef KDA_SYNC_FOR_MMA
#undef KDA_PAIR_MMA
    if (!kSplit && !failed && o_pend) {  // the last chunk's output: all warps, 16 tokens each
        tc::fence_after_sync();
        o_emit(16 * part, 16, true);
        tc::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) o_store();
    }

    if (failed && tid == 0) {
        atomicExch(&g_kda_tc_timeout, 1);
        // give any tensor-core or TMA work still in flight a bounded chance to finish
        tc::mbar_wait(&ms.bar_m0, ph0, 200000000ull);
        tc::mbar_wait(&ms.bar_m1, ph1, 200000000ull);
        tc::mbar_wait(&ms.bar_qkz, ph_qkz, 200000000ull);
        if (!kSplit) tc::mbar_wait(&ms.bar_z, ph_z, 200000000ull);
        tc::mbar_wait(&ms.bar_v, ph_v, 200000000ull);
    }
    if (tid == 0) tc::bulk_wait_all();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

}  // namespace

__global__ void __launch_bounds__(NT, 1)
    kda_chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_z, int H, int T,
                        const __nv_bfloat16* __restrict__ beta, const float* __restrict__ A_log,
                        const float* __restrict__ dt_bias, float scale,
                        const float* __restrict__ h0, __nv_bfloat16* __restrict__ out,
                        float* __restrict__ hT, FusedSched fs) {
    chunk_loop<false>(&tm_q, &tm_k, &tm_v, &tm_z, nullptr, nullptr, nullptr, nullptr, H, T, beta, A_log,
                      dt_bias, scale, h0, out, hT, PrepSeg{0, 1, 0, nullptr, nullptr}, fs);
}

// The chunk-parallel half of the split forward: every chunk of the segment is one work
// item, independent of the state; CTAs take items gridDim.x apart.
__global__ void __launch_bounds__(NT, 1)
    kda_chunk_prep_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_z,
                          const __grid_constant__ CUtensorMap tm_wq,
                          const __grid_constant__ CUtensorMap tm_qg,
                          const __grid_constant__ CUtensorMap tm_uu,
                          const __grid_constant__ CUtensorMap tm_kt, int H, int T,
                          const __nv_bfloat16* __restrict__ beta, const float* __restrict__ A_log,
                          const float* __restrict__ dt_bias, PrepSeg seg) {
    chunk_loop<true>(&tm_q, &tm_k, &tm_v, &tm_z, &tm_wq, &tm_qg, &tm_uu, &tm_kt, H, T, beta, A_log,
                     dt_bias, 0.f, nullptr, nullptr, nullptr, seg,
                     FusedSched{0, 1, 0, nullptr, nullptr, nullptr});
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A driver API entry point, looked up through the runtime (no -lcuda link); null if absent.
void* driver_entry(const char* name) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return p;
}

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = reinterpret_cast<EncodeTiledFn>(driver_entry("cuTensorMapEncodeTiled"));
    return fn;
}

// 3-D bf16 tile map: extents d0 (innermost) .. d2, row pitches s1 / s2 in bytes, box b0 x b1 x 1.
bool make_map3(CUtensorMap* map, const void* base, cuuint64_t d0, cuuint64_t d1, cuuint64_t d2,
               cuuint64_t s1, cuuint64_t s2, cuuint32_t b0, cuuint32_t b1, CUtensorMapSwizzle sw) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {b0, b1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view (channel, token, b*h) of a (B, H, T, 128) bf16 tensor; 64 x 128 tiles, no swizzle.
bool make_tile_map(CUtensorMap* map, const void* base, int T, int BH) {
    return make_map3(map, base, 128, (cuuint64_t)T, (cuuint64_t)BH, 128 * 2, (cuuint64_t)T * 128 * 2,
                     128, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool make_input_maps(const ChunkArgs& a, CUtensorMap (&m)[4]) {
    const int BH = a.B * a.H;
    return make_tile_map(&m[0], a.q, a.T, BH) && make_tile_map(&m[1], a.k, a.T, BH) &&
           make_tile_map(&m[2], a.v, a.T, BH) && make_tile_map(&m[3], a.z, a.T, BH);
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return 1;
    return n;
}

size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

}  // namespace

// Unique id of the CUDA context current on this thread (0 when none is current yet).  A
// device's primary context gets a new id when it is destroyed and created again (after
// cudaDeviceReset); per-device caches of device addresses and CUDA objects compare it to
// notice that what they hold belonged to a context that no longer exists.
cudaError_t current_context_id(unsigned long long* id) {
    typedef CUresult (*GetCurrentFn)(CUcontext*);
    typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = reinterpret_cast<GetCurrentFn>(driver_entry("cuCtxGetCurrent"));
    static GetIdFn get_id = reinterpret_cast<GetIdFn>(driver_entry("cuCtxGetId"));
    *id = 0;
    if (!get_current || !get_id) return cudaErrorNotSupported;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
    if (!ctx) return cudaSuccess;
    return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

// A wait that nothing ever satisfies: one thread initialises an mbarrier that expects one
// arrival, never arrives, and waits with the bounded wait every kernel here uses.  The wait
// gives up after `limit_ns` and records the timeout in the same flag the chunk kernel sets,
// which is how the host-side failure report is exercised without faulting or hanging a GPU.
__global__ void kda_bounded_wait_selftest_kernel(unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_barrier_init();
        if (!tc::mbar_wait(&bar, 0, limit_ns)) atomicExch(&g_kda_tc_timeout, 1);
    }
}

cudaError_t launch_bounded_wait_selftest(unsigned long long limit_ns, cudaStream_t s) {
    kda_bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns);
    count_launches(1);
    return cudaGetLastError();
}

// Reads and clears the timeout flag after the stream has drained; *timed_out = flag.
cudaError_t read_and_clear_timeout(cudaStream_t s, int* timed_out) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_kda_tc_timeout, sizeof(int));
    if (e != cudaSuccess) return e;
    *timed_out = v;
    if (v) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_kda_tc_timeout, &zero, sizeof(int));
    }
    return e;
}

namespace {

bool chunk_tc_eligible(const ChunkArgs& a) {
    return a.io == KDA_BF16 && a.K == 128 && a.V == 128 && a.chunk == 64 && a.T > 0;
}

size_t split_scratch_bytes(const ChunkArgs& a, int seg_len) {
    const size_t BH = (size_t)a.B * a.H;
    return round_up(BH * seg_len * kItemBytes, 256) + (a.hT ? 0 : BH * KD * VD * sizeof(float));
}

// Chunks per segment of the split forward that fit in `bytes` of scratch (0: none fit).
int split_segment_len(const ChunkArgs& a, size_t bytes) {
    const int N = (a.T + C - 1) / C;
    const size_t BH = (size_t)a.B * a.H;
    const size_t state = a.hT ? 0 : BH * KD * VD * sizeof(float);
    if (bytes < state) return 0;
    const size_t per_chunk = BH * kItemBytes;
    size_t len = (bytes - state) / per_chunk;
    if (len > (size_t)N) len = N;
    while (len > 0 && round_up(len * per_chunk, 256) + state > bytes) --len;
    return (int)len;
}

// The per-chunk operands of up to items_max items, carved from p (kItemBytes items_max bytes):
// the [W^T | (Q Gamma)^T], U^T, K~ and M tiles, then Gamma_last, each array item after item.
bool split_operands(uint8_t* p, size_t items_max, SplitOperands* o) {
    uint8_t* wq = p;
    uint8_t* uu = wq + items_max * kItemWQ;
    uint8_t* kt = uu + items_max * kItemUU;
    o->mm = kt + items_max * kItemKT;
    o->gl = reinterpret_cast<float*>(o->mm + items_max * kItemMM);
    return make_map3(&o->wq, wq, 64, 128, 2 * items_max, 128, 16384, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map3(&o->qg, wq, 64, 64, 4 * items_max, 128, 8192, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map3(&o->uu, uu, 64, 128, items_max, 128, 16384, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map3(&o->kt, kt, 128, 64, items_max, 256, 16384, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
}

// The split forward with caller-provided scratch: per segment of chunks, the prep kernel
// (all chunks of all sequences in parallel) then the carry kernel (one CTA per sequence).
cudaError_t run_chunk_split(const ChunkArgs& a, cudaStream_t s, void* scratch, size_t bytes) {
    const int N = (a.T + C - 1) / C, BH = a.B * a.H;
    const int seg_len = split_segment_len(a, bytes);
    if (seg_len < 1) return cudaErrorMemoryAllocation;
    const size_t items_max = (size_t)BH * seg_len;
    uint8_t* p = static_cast<uint8_t*>(scratch);
    float* state = reinterpret_cast<float*>(p + round_up(items_max * kItemBytes, 256));
    CUtensorMap m[4];
    SplitOperands ops;
    if (!make_input_maps(a, m) || !split_operands(p, items_max, &ops)) return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(kda_chunk_prep_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)SMEM_BYTES);
    if (err != cudaSuccess) return err;
    float* h_state = a.hT ? a.hT : state;
    const int nsm = sm_count();
    for (int n0 = 0; n0 < N; n0 += seg_len) {
        const int len = min(seg_len, N - n0), items = BH * len;
        kda_chunk_prep_kernel<<<min(items, nsm), NT, SMEM_BYTES, s>>>(
            m[0], m[1], m[2], m[3], ops.wq, ops.qg, ops.uu, ops.kt, a.H, a.T, (const __nv_bfloat16*)a.beta,
            a.A_log, a.dt_bias, PrepSeg{n0, len, items, ops.mm, ops.gl});
        count_launches(1);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        err = launch_chunk_carry(ops, BH, a.T, n0, len, a.scale, n0 == 0 ? a.h0 : h_state,
                                 (__nv_bfloat16*)a.out, h_state, s);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

// The second stream and the five events of the overlapped split form below: created on the
// first call on a device (and again after that device's context was reset), then kept and
// shared by every call on the device.  A call holds `mu` while it enqueues its work, so no
// other call records the same events in between.
constexpr int kMaxDevices = 64;
struct OverlapRes {
    std::mutex mu;
    unsigned long long ctx = 0;
    cudaStream_t s2 = nullptr;
    cudaEvent_t ev[5] = {};  // fork, prep done [2], carry done [2]
};
OverlapRes g_overlap[kMaxDevices];

// Makes r's stream and events valid for the current context (r.mu held).
cudaError_t overlap_res_ready(OverlapRes& r) {
    unsigned long long ctx = 0;
    cudaError_t err = current_context_id(&ctx);
    if (err != cudaSuccess) return err;
    if (ctx != 0 && ctx == r.ctx) return cudaSuccess;
    // first use, or the objects held belong to a context that is gone: make new ones
    r.ctx = 0;
    r.s2 = nullptr;
    for (cudaEvent_t& e : r.ev) e = nullptr;
    if ((err = cudaStreamCreateWithFlags(&r.s2, cudaStreamNonBlocking)) != cudaSuccess) return err;
    for (cudaEvent_t& e : r.ev)
        if ((err = cudaEventCreateWithFlags(&e, cudaEventDisableTiming)) != cudaSuccess) return err;
    if ((err = current_context_id(&ctx)) != cudaSuccess) return err;
    r.ctx = ctx;
    return cudaSuccess;
}

// The split form with the carry of segment i (one CTA per sequence, on a second stream)
// running beside the prep of segment i + 1 (on the remaining SMs): two operand buffers,
// events between the streams, `s` waits for all of it at the end.  For few sequences
// (B*H at most half the SMs) and two or more segments.
cudaError_t run_chunk_split_overlap(const ChunkArgs& a, cudaStream_t s, void* scratch, int seg_len) {
    const int N = (a.T + C - 1) / C, BH = a.B * a.H, nsm = sm_count();
    const size_t items_max = (size_t)BH * seg_len, buf_bytes = round_up(items_max * kItemBytes, 256);
    CUtensorMap m[4];
    SplitOperands ops[2];
    if (!make_input_maps(a, m)) return cudaErrorInvalidValue;
    for (int b = 0; b < 2; ++b)
        if (!split_operands(static_cast<uint8_t*>(scratch) + b * buf_bytes, items_max, &ops[b]))
            return cudaErrorInvalidValue;
    float* h_state = a.hT ? a.hT
                          : reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + 2 * buf_bytes);
    cudaError_t err = cudaFuncSetAttribute(kda_chunk_prep_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)SMEM_BYTES);
    if (err != cudaSuccess) return err;
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    OverlapRes& res = g_overlap[dev];
    std::lock_guard<std::mutex> lock(res.mu);
    if ((err = overlap_res_ready(res)) != cudaSuccess) return err;
    cudaStream_t s2 = res.s2;
    cudaEvent_t* ev = res.ev;
    err = cudaEventRecord(ev[0], s);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(s2, ev[0], 0);
    const int prep_grid = max(1, nsm - BH);  // leave one SM per carry CTA
    for (int n0 = 0, i = 0; n0 < N && err == cudaSuccess; n0 += seg_len, ++i) {
        const int b = i & 1, len = min(seg_len, N - n0), items = BH * len;
        if (i >= 2) err = cudaStreamWaitEvent(s, ev[3 + b], 0);  // carry of segment i - 2 read buffer b
        if (err != cudaSuccess) break;
        kda_chunk_prep_kernel<<<min(items, prep_grid), NT, SMEM_BYTES, s>>>(
            m[0], m[1], m[2], m[3], ops[b].wq, ops[b].qg, ops[b].uu, ops[b].kt, a.H, a.T,
            (const __nv_bfloat16*)a.beta, a.A_log, a.dt_bias,
            PrepSeg{n0, len, items, ops[b].mm, ops[b].gl});
        count_launches(1);
        if ((err = cudaGetLastError()) != cudaSuccess) break;
        if ((err = cudaEventRecord(ev[1 + b], s)) != cudaSuccess) break;
        if ((err = cudaStreamWaitEvent(s2, ev[1 + b], 0)) != cudaSuccess) break;
        err = launch_chunk_carry(ops[b], BH, a.T, n0, len, a.scale, n0 == 0 ? a.h0 : h_state,
                                 (__nv_bfloat16*)a.out, h_state, s2);
        if (err == cudaSuccess) err = cudaEventRecord(ev[3 + b], s2);
    }
    // join: `s` continues only after the last carry (also on failure, so nothing is left behind)
    const cudaError_t jerr = cudaEventRecord(ev[0], s2) == cudaSuccess
                                 ? cudaStreamWaitEvent(s, ev[0], 0)
                                 : cudaErrorUnknown;
    return err != cudaSuccess ? err : jerr;
}

// Makespan of the overlapped split form (run_chunk_split_overlap) with segments of L chunks,
// the last one shorter, in units of one prep item (one chunk of one sequence on one CTA):
// the prep of a segment of l chunks takes ceil(BH l / G) items on its G CTAs, the carry
// about a fifth of an item per chunk, and each launch about half an item more (measured on
// the B1 H32 and B1 H4 T65536 workloads, about 12 us per item); the prep of segment i starts
// after the prep of i - 1 and the carry of i - 2 (whose operand buffer it overwrites), the
// carry of i after the prep of i and the carry of i - 1.
double overlap_makespan(long long BH, long long N, long long G, long long L) {
    double p_end = 0.0, c_prev = 0.0, c_prev2 = 0.0;
    for (long long n0 = 0; n0 < N; n0 += L) {
        const long long l = std::min(L, N - n0);
        p_end = std::max(p_end, c_prev2) + (double)((BH * l + G - 1) / G) + 0.5;
        const double c = std::max(p_end, c_prev) + 0.2 * (double)l + 0.5;
        c_prev2 = c_prev;
        c_prev = c;
    }
    return c_prev;
}

// Chunks per segment of the overlapped split form: the length of at most `cap` (what the
// scratch allows) with the smallest makespan above, among lengths that make at most 64
// segments of at least 16 chunks where possible.  Lengths whose BH L items fill the prep's
// waves, and a short last segment (a short last carry), come out ahead.  The last answer is
// kept, for calls that repeat a shape.
int overlap_segment_len(long long BH, long long N, long long G, int cap) {
    static thread_local long long last[5] = {-1, -1, -1, -1, -1};
    if (last[0] == BH && last[1] == N && last[2] == G && last[3] == cap) return (int)last[4];
    const long long lo = std::max(16LL, (N + 63) / 64), hi = std::min((long long)cap, N);
    long long best_len = hi;
    if (hi > lo) {
        const long long step = std::max(1LL, (hi - lo) / 256);
        double best = overlap_makespan(BH, N, G, hi);
        for (long long L = lo; L < hi; L += step) {
            const double m = overlap_makespan(BH, N, G, L);
            if (m < best - 1e-9) {
                best = m;
                best_len = L;
            }
        }
    }
    last[0] = BH; last[1] = N; last[2] = G; last[3] = cap; last[4] = best_len;
    return (int)best_len;
}

// Scratch of the allocating split forward: at most this much per call (longer inputs are
// processed in segments of chunks).
constexpr size_t kSplitScratchCap = size_t(1) << 30;

cudaError_t launch_chunk_split(const ChunkArgs& a, cudaStream_t s) {
    const int N = (a.T + C - 1) / C, BH = a.B * a.H, nsm = sm_count();
    // few sequences: two operand buffers and the carry beside the next segment's prep, in
    // segments of the length that the makespan model above picks
    if (2 * BH <= nsm && N >= 4) {
        const int cap = split_segment_len(a, kSplitScratchCap / 2);  // per buffer (and the state)
        const int seg_len = cap >= 1 ? overlap_segment_len(BH, N, nsm - BH, cap) : 0;
        if (seg_len >= 1) {
            const size_t items_max = (size_t)BH * seg_len;
            const size_t bytes = 2 * round_up(items_max * kItemBytes, 256) +
                                 (a.hT ? 0 : (size_t)BH * KD * VD * sizeof(float));
            void* p = nullptr;
            if (scratch_alloc(&p, bytes, s) != cudaSuccess) {
                cudaGetLastError();
                return cudaErrorMemoryAllocation;
            }
            const cudaError_t err = run_chunk_split_overlap(a, s, p, seg_len);
            const cudaError_t ferr = scratch_free(p, s);
            return err != cudaSuccess ? err : ferr;
        }
    }
    const int seg_len = split_segment_len(a, kSplitScratchCap);
    if (seg_len < 1) return cudaErrorMemoryAllocation;
    const size_t bytes = split_scratch_bytes(a, seg_len);
    void* p = nullptr;
    if (scratch_alloc(&p, bytes, s) != cudaSuccess) {
        cudaGetLastError();
        return cudaErrorMemoryAllocation;
    }
    const cudaError_t err = run_chunk_split(a, s, p, bytes);
    const cudaError_t ferr = scratch_free(p, s);
    return err != cudaSuccess ? err : ferr;
}

// Schedule of the fused kernel: *seg_len = chunks per work item (0: one CTA per whole
// sequence) and the cost in chunk steps.  With more sequences than SMs the last wave of whole
// sequences leaves SMs idle; items of a few chunks spread the same work evenly, at about a
// quarter chunk step per item for handing the state on.
double fused_schedule(long long BH, long long N, long long S, int* seg_len) {
    double best = (double)((BH + S - 1) / S) * (double)N;
    *seg_len = 0;
    if (BH <= S) return best;
    for (long long L = N / 2; L >= 2; L /= 2) {
        const long long items = (N + L - 1) / L * BH;
        const double cost = (double)((items + S - 1) / S) * ((double)L + 0.25);
        if (cost < 0.97 * best) {
            best = cost;
            *seg_len = (int)L;
        }
    }
    return best;
}

cudaError_t launch_chunk_fused(const ChunkArgs& a, cudaStream_t s) {
    const int BH = a.B * a.H, N = (a.T + C - 1) / C, nsm = sm_count();
    CUtensorMap m[4];
    if (!make_input_maps(a, m)) return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(kda_chunk_tc_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)SMEM_BYTES);
    if (err != cudaSuccess) return err;
    int L = 0;
    fused_schedule(BH, N, nsm, &L);
    if (L == 0) {  // one CTA per sequence
        kda_chunk_tc_kernel<<<BH, NT, SMEM_BYTES, s>>>(
            m[0], m[1], m[2], m[3], a.H, a.T, (const __nv_bfloat16*)a.beta, a.A_log, a.dt_bias,
            a.scale, a.h0, (__nv_bfloat16*)a.out, a.hT,
            FusedSched{BH, N, BH, nullptr, nullptr, nullptr});
        count_launches(1);
        return cudaGetLastError();
    }
    // items of L chunks taken in order by one CTA per SM: a counter and one flag per sequence
    // (cleared here), and the state between segments in hT (or in scratch when hT is not wanted)
    const int n_items = (N + L - 1) / L * BH;
    const size_t flag_bytes = round_up(sizeof(unsigned) * (1 + (size_t)BH), 256);
    const size_t bytes = flag_bytes + (a.hT ? 0 : (size_t)BH * KD * VD * sizeof(float));
    void* p = nullptr;
    if (scratch_alloc(&p, bytes, s) != cudaSuccess) {
        cudaGetLastError();
        return cudaErrorMemoryAllocation;
    }
    err = cudaMemsetAsync(p, 0, flag_bytes, s);
    if (err == cudaSuccess) {
        unsigned* w = static_cast<unsigned*>(p);
        float* handoff = a.hT ? a.hT : reinterpret_cast<float*>(static_cast<uint8_t*>(p) + flag_bytes);
        kda_chunk_tc_kernel<<<min(n_items, nsm), NT, SMEM_BYTES, s>>>(
            m[0], m[1], m[2], m[3], a.H, a.T, (const __nv_bfloat16*)a.beta, a.A_log, a.dt_bias,
            a.scale, a.h0, (__nv_bfloat16*)a.out, a.hT,
            FusedSched{BH, L, n_items, reinterpret_cast<int*>(w), w + 1, handoff});
        count_launches(1);
        err = cudaGetLastError();
    }
    const cudaError_t ferr = scratch_free(p, s);
    return err != cudaSuccess ? err : ferr;
}

// ---- the split form with the chunk-parallel state scan (few sequences, many chunks)
//
// Sub-segments for a segment of `len` chunks and BH sequences: enough that the carry's Z and P
// roles (2 BH (nsub - 1) CTAs) fill the SMs once, no more than about sqrt(2 len) (the combine
// walks them one by one, a K x K by K x V product each), at least 4 chunks each.
int scan_subsegments(long long BH, long long len, long long S) {
    long long n = S / (2 * BH) + 1;
    n = std::min(n, (long long)std::ceil(std::sqrt(2.0 * (double)len)));
    n = std::min(n, (len + 3) / 4);
    return (int)std::max(1LL, n);
}

// Costs in fused chunk steps (one prep item costs about one; a carry chunk about 0.17 of one):
// the scan form (prep on every SM, then the Z/P roles, the combine and the plain carry over
// the sub-segments), and the overlapped split form (prep beside a carry of one CTA per
// sequence, so bound by the longer of the two).
double scan_cost(long long BH, long long N, long long S) {
    const long long nsub = scan_subsegments(BH, N, S), sub_len = (N + nsub - 1) / nsub;
    const double c = 0.17;
    return (double)((BH * N + S - 1) / S) +
           c * (double)sub_len * (double)((2 * BH * (nsub - 1) + S - 1) / S) + c * (double)nsub +
           c * (double)sub_len * (double)((BH * nsub + S - 1) / S);
}
double split_overlap_cost(long long BH, long long N, long long S) {
    const long long prep_sms = std::max(1LL, S - BH);
    return std::max((double)((BH * N + prep_sms - 1) / prep_sms), 0.17 * (double)N);
}

// Scratch of the scan form for segments of seg_len chunks: the operands of a segment, the
// carried state when hT is not wanted, the Z and P maps of all sub-segments but the last and
// the entering states of all of them.
size_t scan_scratch_bytes(const ChunkArgs& a, int seg_len, int* nsub_max) {
    const size_t BH = (size_t)a.B * a.H, KVB = (size_t)KD * VD * sizeof(float);
    const int nsub = scan_subsegments((long long)BH, seg_len, sm_count());
    *nsub_max = nsub;
    return round_up(BH * seg_len * kItemBytes, 256) + (a.hT ? 0 : round_up(BH * KVB, 256)) +
           2 * round_up((size_t)std::max(1, nsub - 1) * BH * KVB, 256) +
           round_up((size_t)nsub * BH * KVB, 256);
}

cudaError_t run_chunk_split_scan(const ChunkArgs& a, cudaStream_t s, void* scratch, int seg_len,
                                 int nsub_max) {
    const int N = (a.T + C - 1) / C, BH = a.B * a.H, nsm = sm_count();
    const size_t KVB = (size_t)KD * VD * sizeof(float), items_max = (size_t)BH * seg_len;
    uint8_t* p = static_cast<uint8_t*>(scratch);
    size_t off = round_up(items_max * kItemBytes, 256);
    float* state = a.hT;
    if (!state) {
        state = reinterpret_cast<float*>(p + off);
        off += round_up(BH * KVB, 256);
    }
    const size_t map_bytes = round_up((size_t)std::max(1, nsub_max - 1) * BH * KVB, 256);
    float* zbuf = reinterpret_cast<float*>(p + off);
    float* pbuf = reinterpret_cast<float*>(p + off + map_bytes);
    float* sbuf = reinterpret_cast<float*>(p + off + 2 * map_bytes);
    CUtensorMap m[4];
    SplitOperands ops;
    if (!make_input_maps(a, m) || !split_operands(p, items_max, &ops)) return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(kda_chunk_prep_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)SMEM_BYTES);
    if (err != cudaSuccess) return err;
    for (int n0 = 0; n0 < N; n0 += seg_len) {
        const int len = std::min(seg_len, N - n0), items = BH * len;
        kda_chunk_prep_kernel<<<std::min(items, nsm), NT, SMEM_BYTES, s>>>(
            m[0], m[1], m[2], m[3], ops.wq, ops.qg, ops.uu, ops.kt, a.H, a.T, (const __nv_bfloat16*)a.beta,
            a.A_log, a.dt_bias, PrepSeg{n0, len, items, ops.mm, ops.gl});
        count_launches(1);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        const float* h_seg = n0 == 0 ? a.h0 : state;  // entering state of the segment (may be null)
        int nsub = std::min(nsub_max, scan_subsegments(BH, len, nsm));
        const int sub_len = (len + nsub - 1) / nsub;
        nsub = (len + sub_len - 1) / sub_len;
        if (nsub < 2) {
            err = launch_chunk_carry(ops, BH, a.T, n0, len, a.scale, h_seg, (__nv_bfloat16*)a.out,
                                     state, s);
        } else {
            // the maps (P, Z) of sub-segments 0 .. nsub - 2, their entering states in order,
            // then the plain carry of every sub-segment from its entering state
            err = launch_chunk_carry_grid(ops, a.T, n0, len, a.scale, nullptr, nullptr, nullptr,
                                          CarryGrid{BH, nsub - 1, sub_len, 1, zbuf, pbuf}, s);
            if (err == cudaSuccess) err = launch_carry_combine(BH, nsub, h_seg, pbuf, zbuf, sbuf, s);
            if (err == cudaSuccess)
                err = launch_chunk_carry_grid(ops, a.T, n0, len, a.scale, sbuf, (__nv_bfloat16*)a.out,
                                              state, CarryGrid{BH, nsub, sub_len, 0, nullptr, nullptr}, s);
        }
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

cudaError_t launch_chunk_scan(const ChunkArgs& a, cudaStream_t s) {
    const int N = (a.T + C - 1) / C;
    int seg_len = N, nsub_max = 1;
    while (seg_len > 1 && scan_scratch_bytes(a, seg_len, &nsub_max) > kSplitScratchCap)
        seg_len = (seg_len + 1) / 2;
    const size_t bytes = scan_scratch_bytes(a, seg_len, &nsub_max);
    if (bytes > kSplitScratchCap) return cudaErrorMemoryAllocation;
    void* p = nullptr;
    if (scratch_alloc(&p, bytes, s) != cudaSuccess) {
        cudaGetLastError();
        return cudaErrorMemoryAllocation;
    }
    const cudaError_t err = run_chunk_split_scan(a, s, p, seg_len, nsub_max);
    const cudaError_t ferr = scratch_free(p, s);
    return err != cudaSuccess ? err : ferr;
}

// Which tensor-core form is faster: the fused kernel's schedule (above) against the split
// form, which spreads all chunks over the SMs and adds a short sequential carry (about a tenth
// of a fused chunk step) per chunk.
bool prefer_split(const ChunkArgs& a) {
    const long long BH = (long long)a.B * a.H, N = (a.T + C - 1) / C, S = sm_count();
    int L = 0;
    const double fused = fused_schedule(BH, N, S, &L);
    const double split = (double)((BH * N + S - 1) / S) * 0.9 + (double)((BH + S - 1) / S) * N * 0.1;
    return split < 0.85 * fused;
}

}  // namespace

// The split form on caller-provided scratch of `bytes` (no allocation of its own).
// chunk_split_fits: whether the shape takes the split form and one segment of a chunk per
// sequence fits in `bytes`; run_chunk_split_in then runs it.  Every byte of the scratch that
// a call reads, the same call wrote first.
bool chunk_split_fits(const ChunkArgs& a, size_t bytes) {
    return chunk_tc_eligible(a) && split_segment_len(a, bytes) >= 1;
}
cudaError_t run_chunk_split_in(const ChunkArgs& a, cudaStream_t s, void* scratch, size_t bytes) {
    return run_chunk_split(a, s, scratch, bytes);
}

// mode 0: pick the faster form, 1: fused kernel, 2: split form, 3: split form with the
// chunk-parallel state scan.  Mode 0 takes the scan where the overlapped split form would be
// bound by its sequential carry (few sequences over many chunks).
cudaError_t launch_chunk_tc(const ChunkArgs& a, cudaStream_t s, int mode, bool* taken) {
    *taken = false;
    if (!chunk_tc_eligible(a)) return cudaSuccess;
    *taken = true;
    if (mode == 3) return launch_chunk_scan(a, s);
    const bool split = mode == 2 || (mode == 0 && prefer_split(a));
    if (!split) return launch_chunk_fused(a, s);
    if (mode == 0) {
        const long long BH = (long long)a.B * a.H, N = (a.T + C - 1) / C, S = sm_count();
        if (2 * BH <= S && N >= 64 && scan_cost(BH, N, S) < 0.8 * split_overlap_cost(BH, N, S))
            return launch_chunk_scan(a, s);
    }
    return launch_chunk_split(a, s);
}

}  // namespace kda
