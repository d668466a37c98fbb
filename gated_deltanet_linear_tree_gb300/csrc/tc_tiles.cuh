// Lower-triangular [T][T] tile products on tcgen05 tensor cores, shared by
// the series solves beyond the one-launch substitution (the Neumann series
// and the squaring form of the tree closed form, T <= 256, dv = 128).
//
// A [T][T] matrix m (rows and columns are tree nodes, tiles of 64 x 64 on and
// below the diagonal) is staged in shared memory as bf16 hi + lo B operands,
// one 16 KB tile per (r, s <= r): row rho of tile (r, s) is node 64 r + rho,
// its K index node 64 s + j, K-major with the 128-byte swizzle.  The A
// operand is a matrix with 128 columns (value columns, or a group of 128
// columns of another [T][T] matrix) stored transposed in tensor memory as
// bf16 hi + lo: lane = column, block s at columns AY + 64 s (hi 32 columns,
// lo 32).  The fp32 accumulator of block r is at TD + 64 r (lane = column,
// column = node 64 r + rho).  One product pass then computes, for every
// block r,
//     D_r += A_s B_rs^T   for s <= r,
// i.e. the transposed rows 64 r .. 64 r + 63 of m A, with three bf16
// products per tile (hi*hi + hi*lo + lo*hi, fp32 accumulation).
#pragma once

#include "common.cuh"

namespace canopy {
namespace tct {

constexpr int DV = 128;                 // columns of the A operand (tensor-memory lanes)
constexpr int BN = 64;                  // nodes per block
constexpr int MAXNB = kMaxT / BN;       // blocks per tree at most
constexpr int NTILE = MAXNB * (MAXNB + 1) / 2;
constexpr int TILE = 16384;             // hi [64 rows][128 B] then lo
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t AY = 0;              // A operand: block s at 64 s (hi), 64 s + 32 (lo)
constexpr uint32_t TD = 256;            // D: block r at 256 + 64 r

__device__ inline int tile_index(int r, int s) { return r * (r + 1) / 2 + s; }

// Two-part bf16 split with integer operations only: hi = x rounded half-up
// to 8 significant bits, lo = the top 16 bits of x - hi.
__device__ inline uint32_t hi_bits(float x) { return (__float_as_uint(x) + 0x8000u) & 0xFFFF0000u; }
__device__ inline void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const uint32_t h0 = hi_bits(x0), h1 = hi_bits(x1);
    hi = __byte_perm(h0, h1, 0x7632);
    lo = __byte_perm(__float_as_uint(x0 - __uint_as_float(h0)), __float_as_uint(x1 - __uint_as_float(h1)), 0x7632);
}

// Tiles (r, s <= r) of the [T][T] matrix m, times sign, as bf16 hi/lo B
// operands; entries outside the tree read as zero.  nonzero[t] is set for
// every tile t with a nonzero entry (the others contribute nothing and are
// skipped); the caller clears it first.  nt threads take part.
__device__ inline void stage_tiles(uint8_t* sm, const float* m, int T, int nb, float sign, int* nonzero, int nt) {
    constexpr int PER_TILE = BN * 8;  // rows x 16-byte chunks
    constexpr int BATCH = 5;          // chunks whose loads are in flight together
    const int total = nb * (nb + 1) / 2 * PER_TILE;
    for (int e0 = threadIdx.x; e0 < total; e0 += BATCH * nt) {
        float x[BATCH][8];
#pragma unroll
        for (int k = 0; k < BATCH; ++k) {
            const int e = e0 + k * nt;
            const int t = e / PER_TILE, rem = e - t * PER_TILE, rho = rem >> 3, c8 = rem & 7;
            int r = 0;
            while ((r + 1) * (r + 2) / 2 <= t) ++r;
            const int s = t - r * (r + 1) / 2;
            const int i = BN * r + rho, j0 = BN * s + 8 * c8;
            if (e < total && i < T && j0 + 7 < T && (T & 3) == 0) {
                const float4 a = *reinterpret_cast<const float4*>(m + size_t(i) * T + j0);
                const float4 b = *reinterpret_cast<const float4*>(m + size_t(i) * T + j0 + 4);
                x[k][0] = a.x; x[k][1] = a.y; x[k][2] = a.z; x[k][3] = a.w;
                x[k][4] = b.x; x[k][5] = b.y; x[k][6] = b.z; x[k][7] = b.w;
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    x[k][u] = (e < total && i < T && j0 + u < T) ? m[size_t(i) * T + j0 + u] : 0.f;
            }
        }
#pragma unroll
        for (int k = 0; k < BATCH; ++k) {
            const int e = e0 + k * nt;
            if (e >= total) break;
            const int t = e / PER_TILE, rem = e - t * PER_TILE, rho = rem >> 3, c8 = rem & 7;
            bool nz = false;
#pragma unroll
            for (int u = 0; u < 8; ++u) nz |= (x[k][u] != 0.f);
            if (nz) nonzero[t] = 1;  // benign race: every writer stores 1
            uint4 hv, lv;
            split2(sign * x[k][0], sign * x[k][1], hv.x, lv.x);
            split2(sign * x[k][2], sign * x[k][3], hv.y, lv.y);
            split2(sign * x[k][4], sign * x[k][5], hv.z, lv.z);
            split2(sign * x[k][6], sign * x[k][7], hv.w, lv.w);
            uint8_t* base = sm + t * TILE + rho * 128 + ((c8 ^ (rho & 7)) << 4);
            *reinterpret_cast<uint4*>(base) = hv;
            *reinterpret_cast<uint4*>(base + TILE / 2) = lv;
        }
    }
}

// D_r += A_s B_rs^T for every block r < nb and s <= r whose tile has a
// nonzero entry: three bf16 passes (A hi * B hi, A hi * B lo, A lo * B hi),
// K = 64 nodes per tile.
__device__ inline void issue_products(uint32_t tmem, const uint8_t* sm, int nb, const int* nonzero) {
    for (int r = 0; r < nb; ++r)
        for (int s = 0; s <= r; ++s) {
            if (!nonzero[tile_index(r, s)]) continue;
            const uint32_t bt = smem_u32(sm + tile_index(r, s) * TILE);
#pragma unroll
            for (int pass = 0; pass < 3; ++pass) {
                const uint32_t acol = AY + 64 * s + (pass == 2 ? 32 : 0);
                const uint32_t bb = bt + (pass == 1 ? TILE / 2 : 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ts(tmem + TD + 64 * r, tmem + acol + ks * 8, sdesc_sw128(bb + ks * 32),
                                idesc_bf16(128, 64), 1);
            }
        }
}

// 16 values of this thread's lane (x[e] = node n0 + 16 q + e) into D at the
// block's columns as fp32 (with to_d) and into the A operand as bf16 hi/lo
// (with to_a).
__device__ inline void put_chunk(uint32_t lane_base, int n0, int q, const uint32_t (&x)[16], bool to_d, bool to_a) {
    if (to_d) tmem_st16(lane_base + TD + n0 + 16 * q, x);
    if (to_a) {
        uint32_t wh[8], wl[8];
#pragma unroll
        for (int e2 = 0; e2 < 8; ++e2)
            split2(__uint_as_float(x[2 * e2]), __uint_as_float(x[2 * e2 + 1]), wh[e2], wl[e2]);
        tmem_st8(lane_base + AY + n0 + 8 * q, wh);
        tmem_st8(lane_base + AY + n0 + 32 + 8 * q, wl);
    }
}

// Nodes n0 + 16 q .. + 15 of column c of a [B][T][H][DV] array (rows past T
// read as zero).
__device__ inline void load_chunk(uint32_t (&x)[16], const float* src, int b, int h, int T, int H, int n0, int q,
                                  int c) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const int i = n0 + 16 * q + e;
        x[e] = (i < T) ? __float_as_uint(src[((size_t(b) * T + i) * H + h) * DV + c]) : 0u;
    }
}

}  // namespace tct
}  // namespace canopy
