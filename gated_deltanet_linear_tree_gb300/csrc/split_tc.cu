// The split design of the tree verify on tcgen05 tensor cores (bf16 q/k/v,
// dk = dv = 128, T <= 256): the inverse once per (stream, value head), then
// its application.
//
// canopy page (projects.dotslasha.me/p/canopy.md), "Design decisions" (the
// split alternative: (I + G)^-1 built once per (batch, value head) in global
// memory and applied per value tile) and "M4: Solve strategies" (kernel 1
// builds the inverse, kernel 2 applies it).  The inputs are the tensor-core
// Gram's scratch (gram_tc.cu): G and C as [B][H][T][T] fp32 (64 x 64 tiles on
// and below the diagonal, zero off the paths), gamma X_Q and R as
// [B][T][H][dv].
//
// Kernel 1, one CTA of 512 threads per (stream, value head): W = (I + G)^-1
// over G and M = C W over C.  W is lower triangular with the blocks
//     W_r = W_rr (I_r - sum_{s<r} G_rs W_s),   W_rr = (I + G_rr)^-1,
// (W_r the 64 rows of block r, I_r those rows of the identity), built block
// row by block row for a group of 128 of W's columns at a time with
// tc_tiles.cuh's tile product (lane = column j of W): D_r <- I_r^T, then
// D_r += W_s^T (-G_rs)^T for s < r over the staged tiles of -G; D_r is turned
// into the A operand, and D_r <- (that) W_rr^T is a second product whose B
// operand is W_rr, found by substitution along each row's in-block root path
// (W (I + G) = I: rows are independent) from the staged tile of -G_rr.  Then
// M = C W the same way, with the tiles of C staged and A = W^T.
// Kernel 2, one CTA of 512 threads per (stream, value head): with A = R^T,
// U^T = R^T W^T over the staged W tiles, then o^T = gamma X_Q^T + R^T M^T over
// the staged M tiles, o = scale (gamma X_Q + M R).
// All products: three bf16 passes (hi*hi + hi*lo + lo*hi), fp32
// accumulation.  Every mbarrier wait is bounded; a timeout sets
// CANOPY_DEVERR_TIMEOUT, the later steps are skipped, and the products in
// flight are awaited (bounded) before tensor memory is freed.
#include "tc_tiles.cuh"

namespace canopy {

namespace sptc {

using namespace tct;

constexpr int NT = 512;
constexpr int XS = 68;                          // row stride (floats) of the W_rr scratch
constexpr int WSLOT = NTILE * TILE;             // W_rr as a bf16 hi/lo B tile
constexpr int WSCR = WSLOT + TILE;              // W_rr rows, fp32 [64][XS]
constexpr int PLIST = WSCR + BN * XS * 4;       // in-block paths, u8 [64][64]
constexpr int CTRL = PLIST + BN * BN;
constexpr int SMEM = CTRL + 128;
static_assert(SMEM + 1024 <= 227 * 1024, "shared memory");

// State shared by the phases of a CTA: the product barrier and its phase.
struct Sync {
    uint64_t* bar;
    uint32_t phase;
    bool committed;
    int* flag;
};

// Issue (thread 0) what issue(tmem) lays down, commit, and wait everywhere;
// false (for every thread) if the wait gave up.
template <typename F>
__device__ inline bool run(Sync& sy, uint32_t tmem, F issue) {
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        tc_fence_after();
        issue(tmem);
        mma_commit(sy.bar);
    }
    sy.committed = true;
    const bool done = mbar_wait(sy.bar, sy.phase);
    if (!done) *sy.flag = 1;
    sy.phase ^= 1u;
    tc_fence_after();
    return !__syncthreads_or(!done);
}

// D_r += A_a B^T for the one tile at bt (K = 64): three bf16 passes.
__device__ inline void issue_tile(uint32_t tmem, int r, int a, uint32_t bt) {
#pragma unroll
    for (int pass = 0; pass < 3; ++pass) {
        const uint32_t acol = AY + 64 * a + (pass == 2 ? 32 : 0);
        const uint32_t bb = bt + (pass == 1 ? TILE / 2 : 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ts(tmem + TD + 64 * r, tmem + acol + ks * 8, sdesc_sw128(bb + ks * 32), idesc_bf16(128, 64), 1);
    }
}

// The staged tile's entry (row, k) (bf16 hi + lo back to fp32).
__device__ inline float tile_entry(const uint8_t* tile, int row, int k) {
    const int off = row * 128 + (((k >> 3) ^ (row & 7)) << 4) + ((k & 7) << 1);
    const uint32_t hi = *reinterpret_cast<const uint16_t*>(tile + off);
    const uint32_t lo = *reinterpret_cast<const uint16_t*>(tile + TILE / 2 + off);
    return __uint_as_float(hi << 16) + __uint_as_float(lo << 16);
}

// D at the block's 64 columns -> A operand (hi/lo); with zero_d, D <- 0
// after.  Whole warps only.
__device__ inline void d_to_a(uint32_t lane_base, int n0, bool zero_d) {
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
        uint32_t y[16];
        tmem_ld16(lane_base + TD + n0 + 16 * q, y);
        tmem_wait_ld();
        put_chunk(lane_base, n0, q, y, false, true);
        if (zero_d) {
            uint32_t z[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) z[e] = 0u;
            put_chunk(lane_base, n0, q, z, true, false);
        }
    }
}

// Kernel 1: W over G, M over C.
__global__ void __launch_bounds__(NT, 1) invert_tc_kernel(int T, int H, Ws ws) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + CTRL);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + CTRL + 8);
    int* sFlag = reinterpret_cast<int*>(sm + CTRL + 12);
    int* sNz = reinterpret_cast<int*>(sm + CTRL + 16);  // int[NTILE]
    float* sW = reinterpret_cast<float*>(sm + WSCR);
    uint8_t* sPl = sm + PLIST;
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
    const int quad = warp & 3, grp = warp >> 2;   // lane quadrant, node block
    const int c = quad * 32 + (tid & 31);         // tensor-memory lane
    const int nb = (T + BN - 1) / BN;
    const int n0 = BN * grp;
    const size_t bh = size_t(b) * H + h;
    float* Wg = ws.gs + bh * T * T;   // G on entry, W on exit
    float* Mc = ws.cs + bh * T * T;   // C on entry, M on exit

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        *sFlag = 0;
    }
    if (tid < NTILE) sNz[tid] = 0;
    if (warp == 0) {
        tmem_alloc(sTmem, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16);
    Sync sy{bar, 0u, false, sFlag};

    // the tiles of -G (read before any of W is written over G)
    stage_tiles(sm, Wg, T, nb, -1.f, sNz, NT);
    fence_proxy_async_smem();
    __syncthreads();

    bool ok = true;
    const int ngr = (T + DV - 1) / DV;  // groups of 128 columns of W
    for (int g = 0; g < ngr && ok; ++g) {
        const int j = g * DV + c;       // this lane's column of W
        for (int r = 0; r < nb && ok; ++r) {
            if (BN * (r + 1) <= DV * g) {
                // rows above this group's columns: W_r is zero there
                if (grp == r) {
#pragma unroll 1
                    for (int q = 0; q < 4; ++q) {
                        uint32_t z[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) z[e] = 0u;
                        put_chunk(lane_base, n0, q, z, false, true);
                    }
                    tmem_wait_st();
                }
                continue;
            }
            // W_rr into the B slot: thread rho < 64 takes row rho along its
            // in-block path (ascending, rho last), reading G from the staged
            // tile of -G_rr; rows past T stay zero
            if (tid < BN) {
                const int rho = tid, i = BN * r + rho;
                uint64_t bits = 0;
                if (i < T) {
                    const uint32_t* mrow = ws.mask + (size_t(b) * T + i) * ws.W;
                    const uint32_t w0 = mrow[2 * r], w1 = (2 * r + 1 < ws.W) ? mrow[2 * r + 1] : 0u;
                    bits = (uint64_t(w1) << 32 | w0) | (1ull << rho);
                }
                uint8_t* pl = sPl + rho * BN;
                int n = 0;
                for (; bits; bits &= bits - 1) pl[n++] = uint8_t(__ffsll(static_cast<long long>(bits)) - 1);
                const uint8_t* gt = sm + tile_index(r, r) * TILE;
                float* wr = sW + rho * XS;
                for (int e = n - 1; e >= 0; --e) {
                    const int kcol = pl[e];
                    float acc = (e == n - 1) ? 1.f : 0.f;
                    for (int f = e + 1; f < n; ++f) acc += wr[pl[f]] * tile_entry(gt, pl[f], kcol);  // -G staged
                    wr[kcol] = acc;
                }
                uint8_t* bh8 = sm + WSLOT + rho * 128;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    *reinterpret_cast<uint4*>(bh8 + ((c8 ^ (rho & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4*>(bh8 + TILE / 2 + ((c8 ^ (rho & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                }
                for (int e = 0; e < n; ++e) {
                    const int kc = pl[e];
                    const float x = wr[kc];
                    const uint32_t hb = hi_bits(x);
                    const int off = (((kc >> 3) ^ (rho & 7)) << 4) + ((kc & 7) << 1);
                    *reinterpret_cast<uint16_t*>(bh8 + off) = uint16_t(hb >> 16);
                    *reinterpret_cast<uint16_t*>(bh8 + TILE / 2 + off) =
                        uint16_t(__float_as_uint(x - __uint_as_float(hb)) >> 16);
                }
            }
            fence_proxy_async_smem();
            // D_r <- I_r^T (lane j: 1 at row j of block r)
            if (grp == r) {
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t x[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = (j == n0 + 16 * q + e) ? __float_as_uint(1.f) : 0u;
                    put_chunk(lane_base, n0, q, x, true, false);
                }
                tmem_wait_st();
            }
            // D_r += W_s^T (-G_rs)^T, s < r
            ok = run(sy, tmem, [&](uint32_t tm) {
                for (int s = 0; s < r; ++s)
                    if (sNz[tile_index(r, s)]) issue_tile(tm, r, s, smem_u32(sm + tile_index(r, s) * TILE));
            });
            if (!ok) break;
            if (grp == r) {
                d_to_a(lane_base, n0, true);
                tmem_wait_st();
            }
            // D_r <- (I_r - sum G_rs W_s)^T W_rr^T = W_r^T
            ok = run(sy, tmem, [&](uint32_t tm) { issue_tile(tm, r, r, smem_u32(sm + WSLOT)); });
            if (!ok) break;
            if (grp == r) {
                // W_r^T as the A operand of the later rows; W_r over G (the
                // entries j <= i; the rest of the lower triangle is zero)
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t y[16];
                    tmem_ld16(lane_base + TD + n0 + 16 * q, y);
                    tmem_wait_ld();
                    put_chunk(lane_base, n0, q, y, false, true);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int i = n0 + 16 * q + e;
                        if (i < T && j <= i) Wg[size_t(i) * T + j] = __uint_as_float(y[e]);
                    }
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncthreads();  // the B slot and the scratch are free again
        }
    }

    // M = C W, a group of 128 of its columns at a time: A = W^T (the last
    // group's is in place), the tiles of C as B
    if (ok) {
        if (tid < NTILE) sNz[tid] = 0;
        __syncthreads();
        stage_tiles(sm, Mc, T, nb, 1.f, sNz, NT);
        fence_proxy_async_smem();
        for (int g = ngr - 1; g >= 0 && ok; --g) {
            const int j = g * DV + c;
            if (grp < nb) {
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    if (g != ngr - 1) {
                        uint32_t x[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int i = n0 + 16 * q + e;
                            x[e] = (i < T && j <= i) ? __float_as_uint(Wg[size_t(i) * T + j]) : 0u;
                        }
                        put_chunk(lane_base, n0, q, x, false, true);
                    }
                    uint32_t z[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) z[e] = 0u;
                    put_chunk(lane_base, n0, q, z, true, false);
                }
                tmem_wait_st();
            }
            ok = run(sy, tmem, [&](uint32_t tm) { issue_products(tm, sm, nb, sNz); });
            if (!ok) break;
            if (grp < nb) {
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t y[16];
                    tmem_ld16(lane_base + TD + n0 + 16 * q, y);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int i = n0 + 16 * q + e;
                        if (i < T && j <= i) Mc[size_t(i) * T + j] = __uint_as_float(y[e]);
                    }
                }
            }
            __syncthreads();  // this group's columns of M are written
        }
    }
    __syncthreads();
    if (*sFlag && tid == 0) {
        raise_err(ws.err, CANOPY_DEVERR_TIMEOUT);
        if (sy.committed) mbar_wait(bar, sy.phase ^ 1u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// Kernel 2: U = W R into the workspace, o = scale (gamma X_Q + M R).
template <typename OutT>
__global__ void __launch_bounds__(NT, 1) apply_tc_kernel(OutT* __restrict__ o, int T, int H, Ws ws, float scale) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + CTRL);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + CTRL + 8);
    int* sFlag = reinterpret_cast<int*>(sm + CTRL + 12);
    int* sNz = reinterpret_cast<int*>(sm + CTRL + 16);  // int[NTILE]
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
    const int quad = warp & 3, grp = warp >> 2;
    const int c = quad * 32 + (tid & 31);          // value column
    const int nb = (T + BN - 1) / BN;
    const bool active = grp < nb;
    const int n0 = BN * grp;
    const size_t bh = size_t(b) * H + h;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        *sFlag = 0;
    }
    if (tid < NTILE) sNz[tid] = 0;
    if (warp == 0) {
        tmem_alloc(sTmem, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16);
    Sync sy{bar, 0u, false, sFlag};

    // U^T = R^T W^T
    stage_tiles(sm, ws.gs + bh * T * T, T, nb, 1.f, sNz, NT);
    fence_proxy_async_smem();
    if (active) {
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
            uint32_t x[16], z[16];
            load_chunk(x, ws.rr, b, h, T, H, n0, q, c);
#pragma unroll
            for (int e = 0; e < 16; ++e) z[e] = 0u;
            put_chunk(lane_base, n0, q, x, false, true);
            put_chunk(lane_base, n0, q, z, true, false);
        }
        tmem_wait_st();
    }
    bool ok = run(sy, tmem, [&](uint32_t tm) { issue_products(tm, sm, nb, sNz); });
    if (ok && active) {
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
            uint32_t y[16];
            tmem_ld16(lane_base + TD + n0 + 16 * q, y);
            tmem_wait_ld();
            float* up = ws.U + ((size_t(b) * T + n0 + 16 * q) * H + h) * DV + c;
#pragma unroll
            for (int e = 0; e < 16; ++e)
                if (n0 + 16 * q + e < T) up[size_t(e) * H * DV] = __uint_as_float(y[e]);
        }
    }
    // o^T = gamma X_Q^T + R^T M^T
    if (ok) {
        if (tid < NTILE) sNz[tid] = 0;
        __syncthreads();  // (every product of the W tiles has completed)
        stage_tiles(sm, ws.cs + bh * T * T, T, nb, 1.f, sNz, NT);
        fence_proxy_async_smem();
        if (active) {
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t x[16];
                load_chunk(x, ws.xq, b, h, T, H, n0, q, c);
                put_chunk(lane_base, n0, q, x, true, false);
            }
            tmem_wait_st();
        }
        ok = run(sy, tmem, [&](uint32_t tm) { issue_products(tm, sm, nb, sNz); });
        if (ok && active) {
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t y[16];
                tmem_ld16(lane_base + TD + n0 + 16 * q, y);
                tmem_wait_ld();
                OutT* op = o + ((size_t(b) * T + n0 + 16 * q) * H + h) * DV + c;
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (n0 + 16 * q + e < T) store_out(op + size_t(e) * H * DV, scale * __uint_as_float(y[e]));
            }
        }
    }
    __syncthreads();
    if (*sFlag && tid == 0) {
        raise_err(ws.err, CANOPY_DEVERR_TIMEOUT);
        if (sy.committed) mbar_wait(bar, sy.phase ^ 1u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace sptc

// The Gram scratch must be in place (launch_gram_tc); 1 <= T <= 256.
cudaError_t launch_split_tc(int T, int B, int H, void* o, int o_bf16, float scale, const Ws& ws, cudaStream_t st) {
    if (T < 1 || T > kMaxT) return cudaErrorInvalidValue;
    const int smem = sptc::SMEM + 1024;
    dim3 grid(H, B);
    static bool attr_inv = false;
    if (!attr_inv) {
        const cudaError_t e =
            cudaFuncSetAttribute(sptc::invert_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_inv = true;
    }
    sptc::invert_tc_kernel<<<grid, sptc::NT, smem, st>>>(T, H, ws);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (o_bf16) {
        static bool attr = false;
        if (!attr) {
            e = cudaFuncSetAttribute(sptc::apply_tc_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        sptc::apply_tc_kernel<__nv_bfloat16>
            <<<grid, sptc::NT, smem, st>>>(static_cast<__nv_bfloat16*>(o), T, H, ws, scale);
    } else {
        static bool attr = false;
        if (!attr) {
            e = cudaFuncSetAttribute(sptc::apply_tc_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        sptc::apply_tc_kernel<float><<<grid, sptc::NT, smem, st>>>(static_cast<float*>(o), T, H, ws, scale);
    }
    return cudaGetLastError();
}

}  // namespace canopy
