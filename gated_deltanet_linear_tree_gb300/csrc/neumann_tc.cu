// The finite Neumann series of the tree verify on tcgen05 tensor cores, for
// trees of 65 to 256 nodes (bf16 q/k/v, dk = dv = 128).
//
// canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed form"
// and "M4: Solve strategies": G is nilpotent (G^(d+1) = 0 for a tree of depth
// d), so (I + G)^-1 R = sum_{m=0..d} (-G)^m R, d rounds of matrix products on
// tensor cores.  The rounds are taken in Horner's form,
//     Y_0 = R,   Y_{m+1} = R - G Y_m,   U = Y_d,
// which needs one running matrix instead of a running term and a running sum.
// Then o = scale (gamma X_Q + C U).  The inputs are the tensor-core Gram's
// scratch (gram_tc.cu): G and C as [B][H][T][T] fp32 (64 x 64 tiles on and
// below the diagonal, zero off the paths), gamma X_Q and R as [B][T][H][dv].
//
// One CTA of 512 threads per (stream, value head); value columns on the 128
// tensor-memory lanes (the (dv, dk) orientation, D^T = Y^T (-G)^T):
//   tensor memory (512 columns): Y^T as bf16 hi + lo, the A operand of every
//       product (block s at columns 64 s: hi 32 columns, lo 32), and the fp32
//       accumulator D (block r at columns 256 + 64 r);
//   shared memory: the tiles -G_rs (s <= r) as bf16 hi + lo B operands (K-major,
//       128-byte swizzle, 16 KB a tile, at most ten), later the tiles C_rs.
// A round: every thread stores R^T for its 64 nodes into D (R is read once
// and held in registers for all rounds), one thread issues the products
// D_r += Y_s^T (-G_rs)^T for s <= r (bf16 hi*hi + hi*lo + lo*hi, fp32
// accumulation; tiles with no entry on a root path are skipped), and every
// thread turns its part of D into the next Y^T.
// Warp w serves tensor-memory lanes 32 (w % 4) .. + 31 and the 64 nodes of
// block w / 4.  Every mbarrier wait is bounded; a timeout sets
// CANOPY_DEVERR_TIMEOUT, the later rounds are skipped, and the products in
// flight are awaited (bounded) before tensor memory is freed.
#include "tc_tiles.cuh"

namespace canopy {

namespace ntc {

using namespace tct;

constexpr int NT = 512;
constexpr int SMEM = NTILE * TILE + 128;
static_assert(SMEM + 1024 <= 227 * 1024, "shared memory");

// This thread's 64 nodes of a [B][T][H][DV] array (column c) into D.
__device__ inline void load_into_d(uint32_t lane_base, const float* src, int b, int h, int T, int H, int n0, int c) {
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
        uint32_t v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int i = n0 + 16 * q + e;
            v[e] = (i < T) ? __float_as_uint(src[((size_t(b) * T + i) * H + h) * DV + c]) : 0u;
        }
        tmem_st16(lane_base + TD + n0 + 16 * q, v);
    }
    tmem_wait_st();
}

template <typename OutT>
__global__ void __launch_bounds__(NT, 1) neumann_tc_kernel(OutT* __restrict__ o, int T, int H, Ws ws, float scale) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + NTILE * TILE);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + NTILE * TILE + 8);
    int* sDepth = reinterpret_cast<int*>(sm + NTILE * TILE + 12);
    int* sFlag = reinterpret_cast<int*>(sm + NTILE * TILE + 16);
    int* sNz = reinterpret_cast<int*>(sm + NTILE * TILE + 32);  // int[NTILE]
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
    const int quad = warp & 3, grp = warp >> 2;   // lane quadrant, node block
    const int c = quad * 32 + (tid & 31);         // value column (tensor-memory lane)
    const int nb = (T + BN - 1) / BN;
    const bool active = grp < nb;                 // this warp's node block exists
    const int n0 = BN * grp;
    const size_t bh = size_t(b) * H + h;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        *sDepth = 0;
        *sFlag = 0;
        for (int t = 0; t < NTILE; ++t) sNz[t] = 0;
    }
    if (warp == 0) {
        tmem_alloc(sTmem, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16);
    // the stream's depth d (tree prep's depths): G^(d+1) = 0
    for (int i = tid; i < T; i += NT) atomicMax(sDepth, ws.depth[size_t(b) * T + i]);
    stage_tiles(sm, ws.gs + bh * T * T, T, nb, -1.f, sNz, NT);
    fence_proxy_async_smem();
    __syncthreads();
    const int d = min(max(*sDepth, 0), T - 1);

    // Y_0 = R: R^T into D, then into the A operand as hi/lo (the same pass
    // as every later round's conversion); this thread's 64 entries of R stay
    // in registers
    uint32_t phase = 0;   // parity of the next commit's phase
    bool committed = false;
    uint32_t rv[4][16];
    if (active) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int i = n0 + 16 * q + e;
                rv[q][e] = (i < T) ? __float_as_uint(ws.rr[((size_t(b) * T + i) * H + h) * DV + c]) : 0u;
            }
    }
    for (int m = 0; m <= d; ++m) {
        if (active) {  // D <- R^T
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_st16(lane_base + TD + n0 + 16 * q, rv[q]);
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();
        if (m > 0) {
            // D_r = R^T_r + sum_{s <= r} Y_s^T (-G_rs)^T
            if (tid == 0) {
                tc_fence_after();
                issue_products(tmem, sm, nb, sNz);
                mma_commit(bar);
            }
            committed = true;
            if (!mbar_wait(bar, phase)) *sFlag = 1;
            phase ^= 1u;
            tc_fence_after();
        }
        // D (Y_m) -> Y^T hi/lo for the next round; the last round's D is U
        if (active) {
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {  // 16 nodes: hi and lo columns n0 + 8 q (+ 32)
                uint32_t y[16], wh[8], wl[8];
                tmem_ld16(lane_base + TD + n0 + 16 * q, y);
                tmem_wait_ld();
#pragma unroll
                for (int e2 = 0; e2 < 8; ++e2)
                    split2(__uint_as_float(y[2 * e2]), __uint_as_float(y[2 * e2 + 1]), wh[e2], wl[e2]);
                tmem_st8(lane_base + AY + n0 + 8 * q, wh);
                tmem_st8(lane_base + AY + n0 + 32 + 8 * q, wl);
                if (m == d) {
                    float* up = ws.U + ((size_t(b) * T + n0 + 16 * q) * H + h) * DV + c;
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (n0 + 16 * q + e < T) up[size_t(e) * H * DV] = __uint_as_float(y[e]);
                }
            }
            tmem_wait_st();
        }
        tc_fence_before();
        if (__syncthreads_or(*sFlag)) break;
    }

    // o = scale (gamma X_Q + C U): C tiles in place of -G, D <- gamma X_Q^T,
    // D_r += U_s^T C_rs^T
    if (!*sFlag) {
        if (tid < NTILE) sNz[tid] = 0;
        __syncthreads();
        stage_tiles(sm, ws.cs + bh * T * T, T, nb, 1.f, sNz, NT);
        fence_proxy_async_smem();
        if (active) load_into_d(lane_base, ws.xq, b, h, T, H, n0, c);
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            issue_products(tmem, sm, nb, sNz);
            mma_commit(bar);
        }
        committed = true;
        const bool done = mbar_wait(bar, phase);
        if (!done) *sFlag = 1;
        phase ^= 1u;
        tc_fence_after();
        if (active && done) {
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
        // a wait gave up: let the last products issued finish (bounded)
        // before tensor memory is freed
        raise_err(ws.err, CANOPY_DEVERR_TIMEOUT);
        if (committed) mbar_wait(bar, phase ^ 1u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace ntc

// The Gram scratch must be in place (launch_gram_tc); 64 < T <= 256.
cudaError_t launch_neumann_tc(int T, int B, int H, void* o, int o_bf16, float scale, const Ws& ws, cudaStream_t st) {
    if (T <= ntc::BN || T > kMaxT) return cudaErrorInvalidValue;
    const int smem = ntc::SMEM + 1024;
    dim3 grid(H, B);
    if (o_bf16) {
        static bool attr = false;
        if (!attr) {
            const cudaError_t e = cudaFuncSetAttribute(ntc::neumann_tc_kernel<__nv_bfloat16>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        ntc::neumann_tc_kernel<__nv_bfloat16>
            <<<grid, ntc::NT, smem, st>>>(static_cast<__nv_bfloat16*>(o), T, H, ws, scale);
    } else {
        static bool attr = false;
        if (!attr) {
            const cudaError_t e = cudaFuncSetAttribute(ntc::neumann_tc_kernel<float>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        ntc::neumann_tc_kernel<float><<<grid, ntc::NT, smem, st>>>(static_cast<float*>(o), T, H, ws, scale);
    }
    return cudaGetLastError();
}

}  // namespace canopy
