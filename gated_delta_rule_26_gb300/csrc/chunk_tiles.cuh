// chunk_tiles.cuh -- tile geometry shared by the tensor-core chunk kernels (K = V = 128,
// chunk C = 64, bf16 operands): element offsets in the tcgen05 canonical 128-byte-swizzled
// layouts, operand descriptors, TMEM addressing and bf16 packing.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "tc_ptx.cuh"

namespace kda {
namespace tile {

constexpr int C = 64, KD = 128, VD = 128;

// Bytes of the per-chunk operands the chunk-parallel prep kernel hands to the carry kernel:
// W^T (128 x 64 bf16, MN-major) and Q Gamma (64 x 128 bf16, K-major), U^T (128 x 64 bf16),
// K~ (64 x 128 bf16), M (64 x 64 bf16, the masked Q K products of the output) and Gamma_last
// (128 fp32).
constexpr size_t kItemWQ = 2u * 128u * 64u * 2u;
constexpr size_t kItemUU = 128u * 64u * 2u;
constexpr size_t kItemKT = 64u * 128u * 2u;
constexpr size_t kItemMM = 64u * 64u * 2u;
constexpr size_t kItemGL = 128u * 4u;
constexpr size_t kItemBytes = kItemWQ + kItemUU + kItemKT + kItemMM + kItemGL;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ void unpack8(uint4 r, float (&f)[8]) {
    f[0] = bf_lo(r.x); f[1] = bf_hi(r.x); f[2] = bf_lo(r.y); f[3] = bf_hi(r.y);
    f[4] = bf_lo(r.z); f[5] = bf_hi(r.z); f[6] = bf_lo(r.w); f[7] = bf_hi(r.w);
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(tc::pack_bf16x2(f[0], f[1]), tc::pack_bf16x2(f[2], f[3]),
                      tc::pack_bf16x2(f[4], f[5]), tc::pack_bf16x2(f[6], f[7]));
}

// Eight bf16 values (a uint4) times eight factors: the factors are rounded to bf16 pairwise and
// each product, formed by the packed bf16x2 multiply, is rounded to bf16 once.
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint4 scale8_bf16(uint4 x, const float (&f)[8]) {
    return make_uint4(mul_bf16x2(x.x, tc::pack_bf16x2(f[0], f[1])),
                      mul_bf16x2(x.y, tc::pack_bf16x2(f[2], f[3])),
                      mul_bf16x2(x.z, tc::pack_bf16x2(f[4], f[5])),
                      mul_bf16x2(x.w, tc::pack_bf16x2(f[6], f[7])));
}

// K-major tile with `rows` rows: byte offset of element (row, k); k atoms of 64.
__device__ __forceinline__ uint32_t kmaj_off(int row, int k, int rows) {
    return (uint32_t)((k >> 6) * (rows * 128)) + tc::sw128_offset(row, (k & 63) >> 3) + (k & 7) * 2;
}
// MN-major tile: element (krow, mn), MN atoms of 64 elements `atom` bytes apart.
__device__ __forceinline__ uint32_t mnmaj_off(int krow, int mn, uint32_t atom) {
    return (uint32_t)(mn >> 6) * atom + tc::sw128_offset(krow, (mn & 63) >> 3) + (mn & 7) * 2;
}
// 16 consecutive elements (two 16-byte chunks) of one row of a K-major / MN-major tile.
__device__ __forceinline__ void store16_k(uint8_t* base, int row, int k0, int rows, const float (&f)[16]) {
    float lo[8], hi[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) { lo[j] = f[j]; hi[j] = f[8 + j]; }
    *reinterpret_cast<uint4*>(base + kmaj_off(row, k0, rows)) = pack8(lo);
    *reinterpret_cast<uint4*>(base + kmaj_off(row, k0 + 8, rows)) = pack8(hi);
}
__device__ __forceinline__ void store16_mn(uint8_t* base, int krow, int mn0, uint32_t atom, const float (&f)[16]) {
    float lo[8], hi[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) { lo[j] = f[j]; hi[j] = f[8 + j]; }
    *reinterpret_cast<uint4*>(base + mnmaj_off(krow, mn0, atom)) = pack8(lo);
    *reinterpret_cast<uint4*>(base + mnmaj_off(krow, mn0 + 8, atom)) = pack8(hi);
}
// 16 consecutive elements of row `row` of a K-major tile, as fp32.
__device__ __forceinline__ void load16_k(const uint8_t* base, int row, int k0, int rows, float (&f)[16]) {
    float lo[8], hi[8];
    unpack8(*reinterpret_cast<const uint4*>(base + kmaj_off(row, k0, rows)), lo);
    unpack8(*reinterpret_cast<const uint4*>(base + kmaj_off(row, k0 + 8, rows)), hi);
#pragma unroll
    for (int j = 0; j < 8; ++j) { f[j] = lo[j]; f[8 + j] = hi[j]; }
}
// Descriptors of the 16-element K step `ks` of a tile at `saddr`.  The start address sits in
// the descriptor's low bits (in 16-byte units, 14 bits: shared addresses stay below 256 KB), so
// a step's descriptor is the tile's plus a constant: one base per tile, then additions.
__device__ __forceinline__ uint64_t desc_k(uint32_t saddr, int rows, int ks) {
    const int k0 = ks * 16;
    const uint32_t off = (uint32_t)((k0 >> 6) * (rows * 128) + (k0 & 63) * 2);
    return tc::smem_desc(saddr, 16, 1024) + (uint64_t)(off >> 4);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t saddr, uint32_t atom, int ks) {
    return tc::smem_desc(saddr, atom, 1024) + (uint64_t)(ks * (2048 >> 4));
}
// Row-major bf16 output from a lane-per-column layout: lane l of a warp holds o[t][v] for one
// column v (v even on even lanes) and the 16 tokens t = t0 + i.  Neighbouring lanes swap one
// value per token pair, so each lane writes 32-bit pairs (v, v + 1): even lanes the even
// tokens, odd lanes the odd ones.  Rows at or beyond `rows` are not written.
__device__ __forceinline__ void store_o16_pairs(__nv_bfloat16* out_t0, int v, int lane, int rows,
                                                const float (&o)[16]) {
    const bool odd = (lane & 1) != 0;
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float send = odd ? o[i] : o[i + 1];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
        const int t = odd ? i + 1 : i;
        const uint32_t pr = odd ? tc::pack_bf16x2(recv, o[i + 1]) : tc::pack_bf16x2(o[i], recv);
        if (t < rows)
            *reinterpret_cast<uint32_t*>(out_t0 + (size_t)t * VD + (v & ~1)) = pr;
    }
}

// TMEM address of lane quarter (warp & 3) at column `col`.
__device__ __forceinline__ uint32_t taddr(uint32_t base, int warp, uint32_t col) {
    return base + ((uint32_t)((warp & 3) * 32) << 16) + col;
}

}  // namespace tile

// Host side of the split forward's carry kernel (chunk_carry.cu).  SplitOperands: where the
// prep kernel left a segment's per-chunk operands (item = bh * seg_len + chunk of the
// segment): tile maps of W^T (z = 2 item) and, over the same array, of Q Gamma's two 64-channel
// atoms (z = 4 item + 2, 4 item + 3), of U^T (z = item) and K~ (z = item), and the M tiles
// (mm + kItemMM item, the bytes of the shared-memory tile) and Gamma_last (gl + 128 item) as
// plain arrays.
struct SplitOperands {
    CUtensorMap wq, qg, uu, kt;
    uint8_t* mm;
    float* gl;
};
// CarryGrid: BH sequences x nsub sub-segments of sub_len chunks per launch; with scan_roles
// the grid doubles into the scan's Z role (from S = 0, into zbuf) and P role (from the
// identity with U = 0, into pbuf), both laid out [sub][bh][K][V] and neither writing o.
struct CarryGrid {
    int BH, nsub, sub_len, scan_roles;
    float* zbuf;
    float* pbuf;
};
cudaError_t launch_chunk_carry_grid(const SplitOperands& ops, int T, int seg_n0, int seg_len,
                                    float scale, const float* h_in, __nv_bfloat16* out,
                                    float* h_out, const CarryGrid& cg, cudaStream_t s);
cudaError_t launch_carry_combine(int BH, int nsub, const float* h_in, const float* pbuf,
                                 const float* zbuf, float* s_out, cudaStream_t s);
cudaError_t launch_chunk_carry(const SplitOperands& ops, int BH, int T, int seg_n0, int seg_len,
                               float scale, const float* h_in, __nv_bfloat16* out, float* h_out,
                               cudaStream_t s);
cudaError_t read_and_clear_carry_timeout(int* timed_out);

}  // namespace kda
