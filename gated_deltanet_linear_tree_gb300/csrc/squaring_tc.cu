// The squaring form of the tree closed form on tcgen05 tensor cores (bf16
// q/k/v, dk = dv = 128, T <= 256).
//
// canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed form"
// and "M4: Solve strategies": G is nilpotent (G^(d+1) = 0 for a tree of
// depth d), so
//     (I + G)^-1 = (I - G)(I + G^2)(I + G^4) ... (I + G^(2^(k-1))),
// k the least integer with 2^k >= d + 1 (no factor for d = 0).  Taken right
// to left on Z = R:
//     Z <- (I - G) Z;   then for f = 1 .. k - 1:  P <- P^2 (P = G^(2^f)),
//                                                Z <- (I + P) Z;
// U = Z, and o = scale (gamma X_Q + C U).  The inputs are the tensor-core
// Gram's scratch (gram_tc.cu): G and C as [B][H][T][T] fp32 (64 x 64 tiles
// on and below the diagonal, zero off the paths), gamma X_Q and R as
// [B][T][H][dv].  The powers of G overwrite G in place and Z lives in the
// workspace's U between factors.
//
// One CTA of 512 threads per (stream, value head).  Every product is one
// pass of tc_tiles.cuh's lower-triangular tile product D_r += A_s B_rs^T
// (three bf16 products per tile, fp32 accumulation), with the tiles of
// sign P staged in shared memory as B:
//   Z <- Z + sign P Z:  A = Z^T (lane = value column), D starts as Z^T;
//   P^2:                A = (sign P)^T restricted to a group of 128 of P's
//                       columns (lane = column j), D starts at zero and ends
//                       as (P^2)^T for those columns: lane j, column i holds
//                       (P^2)_ij, written back to the [T][T] scratch.
// Warp w serves tensor-memory lanes 32 (w % 4) .. + 31 and the 64 nodes of
// block w / 4.  Every mbarrier wait is bounded; a timeout sets
// CANOPY_DEVERR_TIMEOUT, the later steps are skipped, and the products in
// flight are awaited (bounded) before tensor memory is freed.
#include "tc_tiles.cuh"

namespace canopy {

namespace sqtc {

using namespace tct;

constexpr int NT = 512;
constexpr int SMEM = NTILE * TILE + 128;
static_assert(SMEM + 1024 <= 227 * 1024, "shared memory");

template <typename OutT>
__global__ void __launch_bounds__(NT, 1) squaring_tc_kernel(OutT* __restrict__ o, int T, int H, Ws ws, float scale) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + NTILE * TILE);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + NTILE * TILE + 8);
    int* sDepth = reinterpret_cast<int*>(sm + NTILE * TILE + 12);
    int* sFlag = reinterpret_cast<int*>(sm + NTILE * TILE + 16);
    int* sNz = reinterpret_cast<int*>(sm + NTILE * TILE + 32);  // int[NTILE]
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
    const int quad = warp & 3, grp = warp >> 2;   // lane quadrant, node block
    const int c = quad * 32 + (tid & 31);         // tensor-memory lane
    const int nb = (T + BN - 1) / BN;
    const bool active = grp < nb;                 // this warp's node block exists
    const int n0 = BN * grp;
    const size_t bh = size_t(b) * H + h;
    float* P = ws.gs + bh * T * T;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        *sDepth = 0;
        *sFlag = 0;
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
    __syncthreads();
    const int d = min(max(*sDepth, 0), T - 1);
    int k = 0;
    while ((1 << k) < d + 1) ++k;

    uint32_t phase = 0;   // parity of the next commit's phase
    bool committed = false;
    // one product pass over the staged tiles; false if its wait gave up
    auto run_products = [&]() -> bool {
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
        return !__syncthreads_or(!done);
    };
    auto stage = [&](const float* m, float sign) {
        if (tid < NTILE) sNz[tid] = 0;
        __syncthreads();
        stage_tiles(sm, m, T, nb, sign, sNz, NT);
        fence_proxy_async_smem();
    };

    // Z = R (U = R when there is no factor)
    const float* zsrc = ws.rr;
    bool ok = true;
    for (int f = 0; f < k && ok; ++f) {
        const float sign = f == 0 ? -1.f : 1.f;
        stage(P, sign);
        // Z <- Z + sign P Z
        if (active) {
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t x[16];
                load_chunk(x, zsrc, b, h, T, H, n0, q, c);
                put_chunk(lane_base, n0, q, x, true, true);
            }
            tmem_wait_st();
        }
        ok = run_products();
        if (!ok) break;
        if (active) {
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
        zsrc = ws.U;
        if (f + 1 == k) break;
        // P <- P^2 (sign P times (sign P)^T's transpose), a group of 128 of
        // its columns at a time; the staged tiles still hold sign P, and a
        // group's result overwrites only its own columns of the scratch
        for (int g = 0; g * DV < T && ok; ++g) {
            const int j = g * DV + c;  // this lane's column of P
            if (active) {
                // __syncthreads in run_products orders these reads of P
                // before any thread's write of this group's columns
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t x[16], z[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int i = n0 + 16 * q + e;
                        // P is strictly lower triangular (only strict
                        // ancestors); the scratch above the diagonal tiles
                        // is never written, so it is not read either
                        x[e] = (i < T && j < i) ? __float_as_uint(sign * P[size_t(i) * T + j]) : 0u;
                        z[e] = 0u;
                    }
                    put_chunk(lane_base, n0, q, z, true, false);
                    put_chunk(lane_base, n0, q, x, false, true);
                }
                tmem_wait_st();
            }
            ok = run_products();
            if (!ok) break;
            // (the whole warp reads the accumulator: tcgen05.ld is a
            // warp-wide instruction; lanes past T only skip the stores)
            if (active) {
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t y[16];
                    tmem_ld16(lane_base + TD + n0 + 16 * q, y);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int i = n0 + 16 * q + e;
                        if (i < T && j < i) P[size_t(i) * T + j] = __uint_as_float(y[e]);
                    }
                }
            }
            __syncthreads();  // this group's columns are written before the next group reads P
        }
    }

    // o = scale (gamma X_Q + C U): C tiles, A = U^T, D <- gamma X_Q^T
    if (ok) {
        if (k == 0 && active) {
            // no factor: U = R
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t x[16];
                load_chunk(x, ws.rr, b, h, T, H, n0, q, c);
                float* up = ws.U + ((size_t(b) * T + n0 + 16 * q) * H + h) * DV + c;
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (n0 + 16 * q + e < T) up[size_t(e) * H * DV] = __uint_as_float(x[e]);
            }
        }
        __syncthreads();  // U is in the workspace
        stage(ws.cs + bh * T * T, 1.f);
        if (active) {
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t x[16];
                load_chunk(x, ws.U, b, h, T, H, n0, q, c);
                put_chunk(lane_base, n0, q, x, false, true);
                load_chunk(x, ws.xq, b, h, T, H, n0, q, c);
                put_chunk(lane_base, n0, q, x, true, false);
            }
            tmem_wait_st();
        }
        ok = run_products();
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
        // a wait gave up: let the last products issued finish (bounded)
        // before tensor memory is freed
        raise_err(ws.err, CANOPY_DEVERR_TIMEOUT);
        if (committed) mbar_wait(bar, phase ^ 1u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace sqtc

// The Gram scratch must be in place (launch_gram_tc); 1 <= T <= 256.
cudaError_t launch_squaring_tc(int T, int B, int H, void* o, int o_bf16, float scale, const Ws& ws, cudaStream_t st) {
    if (T < 1 || T > kMaxT) return cudaErrorInvalidValue;
    const int smem = sqtc::SMEM + 1024;
    dim3 grid(H, B);
    if (o_bf16) {
        static bool attr = false;
        if (!attr) {
            const cudaError_t e = cudaFuncSetAttribute(sqtc::squaring_tc_kernel<__nv_bfloat16>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        sqtc::squaring_tc_kernel<__nv_bfloat16>
            <<<grid, sqtc::NT, smem, st>>>(static_cast<__nv_bfloat16*>(o), T, H, ws, scale);
    } else {
        static bool attr = false;
        if (!attr) {
            const cudaError_t e = cudaFuncSetAttribute(sqtc::squaring_tc_kernel<float>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        sqtc::squaring_tc_kernel<float><<<grid, sqtc::NT, smem, st>>>(static_cast<float*>(o), T, H, ws, scale);
    }
    return cudaGetLastError();
}

}  // namespace canopy
