// Gram products of the tree verify on tcgen05 tensor cores (bf16 q/k/v,
// fp32 S0, fp32 accumulation in tensor memory), written to the workspace as
// the inputs of the solve variants in solve_variants.cu (the Neumann series
// beyond one 64-node block, the squaring form and the split design).
//
// canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed form"
// (Bole's Theorem 1), in the (dv, dk) orientation:
//     X_Q = Q S0^T,  X_K = K S0^T,
//     R_i = beta_i (v_i - gamma_i X_K,i),
//     G_ij = beta_i exp(l_i - l_j) k_i.k_j   (j a strict ancestor of i),
//     C_ij = exp(l_i - l_j) q_i.k_j          (j on path(i), i included),
// and "Design decisions" (64-node blocks; the T x T products blocked as
// 64 x 64 tiles, only the tiles on or below the diagonal, since ancestors
// come first in a topological order).
//
// One CTA (256 threads) per (stream b, head h, 64-node row block r), in two
// phases that share 256 tensor-memory columns and 84 KB of shared memory, so
// that two CTAs fit on an SM:
//   1. S0 (fp32) passes box by box through a two-slot staging area and is
//      split into bf16 hi + lo pairs in tensor memory (the A operand); one
//      thread issues X^T = S0 [Q_r; K_r]^T (value columns on the lanes, two
//      products, Q_r and K_r by TMA with the 128-byte swizzle); all eight
//      warps (a lane per value column, two warps per lane, each with half of
//      a box and then half of the nodes) convert S0 and write gamma X_Q and
//      R for the block's nodes;
//   2. the earlier K_s (s < r) come by TMA into the freed staging area; one
//      thread issues [Q_r; K_r] K_s^T for s = 0..r (M = 128, N = 64) into the
//      freed columns; all eight warps (two per row of [Q_r; K_r], tiles
//      shared between them) apply the path mask, the decay and beta and
//      write the C or G row segments.
// Every wait is bounded.
#include "common.cuh"

namespace canopy {

namespace gtc {

constexpr int DV = 128;   // value columns (dk = dv = 128)
constexpr int TP = 64;    // nodes per block
constexpr int NT = 256;   // threads per CTA
constexpr int MAXB = kMaxT / TP;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t TA = 0;     // phase 1: S0 as A: hi [0,64), lo [64,128)
constexpr uint32_t TX = 128;   // phase 1: X^T: Q part [128,192), K part [192,256)
constexpr uint32_t TG = 0;     // phase 2: [Q_r; K_r] K_s^T: block s at [64 s, 64 s + 64)

struct Smem {
    static constexpr int QK = 0;                        // [Q_r; K_r] bf16: 2 key atoms x 128 rows x 128 B
    static constexpr int S0S = 32768;                   // phase 1: S0 staging, two boxes of [128 rows][32 cols]
    static constexpr int S0_BOX = 16384;
    static constexpr int VT = S0S + 2 * S0_BOX;          // phase 1: V_r bf16: 2 tiles [64 nodes][64 cols]
    static constexpr int V_TILE = 8192;
    static constexpr int KS = S0S;                      // phase 2: K_s (s < r), 2 key atoms x 64 rows x 128 B each
    static constexpr int KS_TILE = 16384;
    static constexpr int LL = VT + 2 * V_TILE;           // float[kMaxT]: l of head h for every node
    static constexpr int BG = LL + kMaxT * 4;            // float2[64]: (beta, gamma) of block r's nodes
    static constexpr int MASKW = BG + TP * 8;            // u32[64][8]: strict-ancestor words of block r's nodes
    static constexpr int BAR = MASKW + TP * 8 * 4;       // u64[8]
    static constexpr int TMEMSLOT = BAR + 64;
    static constexpr int FLAG = TMEMSLOT + 4;
    static constexpr int TOTAL = FLAG + 4;
    static_assert(S0S % 1024 == 0 && VT % 1024 == 0 && BAR % 8 == 0, "align");
    static_assert(KS + (MAXB - 1) * KS_TILE <= LL, "the K_s tiles fit the phase-1 area");
    static_assert(TOTAL + 1024 <= 113 * 1024, "two CTAs per SM");
};

enum { BAR_QK = 0, BAR_KS, BAR_V, BAR_S0, BAR_S0B, BAR_AC, BAR_X, NBAR };
static_assert(NBAR <= 8 && BAR_S0B == BAR_S0 + 1, "barriers");

// Two-part bf16 split with integer operations only: hi = x rounded half-up to
// 8 significant bits, lo = the top 16 bits of x - hi (exact in fp32).
__device__ inline uint32_t hi_bits(float x) { return (__float_as_uint(x) + 0x8000u) & 0xFFFF0000u; }
__device__ inline uint32_t pack_top(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632); }
__device__ inline void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const uint32_t h0 = hi_bits(x0), h1 = hi_bits(x1);
    hi = pack_top(h0, h1);
    lo = pack_top(__float_as_uint(x0 - __uint_as_float(h0)), __float_as_uint(x1 - __uint_as_float(h1)));
}

__global__ void __launch_bounds__(NT, 2)
    gram_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmS,
                   const float* __restrict__ beta, int T, int H, int HK, Ws ws) {
    using L = Smem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + L::TMEMSLOT);
    int* sFlag = reinterpret_cast<int*>(sm + L::FLAG);
    float* sL = reinterpret_cast<float*>(sm + L::LL);
    float2* sBG = reinterpret_cast<float2*>(sm + L::BG);
    uint32_t* sMask = reinterpret_cast<uint32_t*>(sm + L::MASKW);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3;  // TMEM lane quadrant of this warp
    const int r = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int n0 = TP * r;      // first node of the block
    const int hk = h / (H / HK);  // the key head this value head reads
    uint8_t* sQK = sm + L::QK;

    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        *sFlag = 0;
        mbar_expect_tx(&bars[BAR_QK], 4 * TP * 64 * 2);
        tma_load_4d(sQK + 0, &tmQ, &bars[BAR_QK], 0, hk, n0, b);
        tma_load_4d(sQK + 16384, &tmQ, &bars[BAR_QK], 64, hk, n0, b);
        tma_load_4d(sQK + 8192, &tmK, &bars[BAR_QK], 0, hk, n0, b);
        tma_load_4d(sQK + 24576, &tmK, &bars[BAR_QK], 64, hk, n0, b);
        for (int i = 0; i < 2; ++i) {
            mbar_expect_tx(&bars[BAR_S0 + i], L::S0_BOX);
            tma_load_4d(sm + L::S0S + i * L::S0_BOX, &tmS, &bars[BAR_S0 + i], 32 * i, 0, h, b);
        }
        mbar_expect_tx(&bars[BAR_V], 2 * L::V_TILE);
        tma_load_4d(sm + L::VT, &tmV, &bars[BAR_V], 0, h, n0, b);
        tma_load_4d(sm + L::VT + L::V_TILE, &tmV, &bars[BAR_V], 64, h, n0, b);
    }
    if (warp == 0) {
        tmem_alloc(sTmem, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    // l of head h for every node (written by tree prep, natural log)
    for (int j = tid; j < T; j += NT) sL[j] = ws.l[(size_t(b) * T + j) * H + h];
    __syncthreads();
    if (tid < TP) {
        const int i = n0 + tid;
        float be = 0.f, gm = 1.f;
        if (i < T) {
            be = beta[(size_t(b) * T + i) * H + h];
            gm = expf(sL[i]);
        }
        sBG[tid] = make_float2(be, gm);
        for (int w = 0; w < 8; ++w)
            sMask[tid * 8 + w] = (i < T && w < ws.W) ? ws.mask[(size_t(b) * T + i) * ws.W + w] : 0u;
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16);

    // ---- phase 1 (all eight warps; warps w and w + 4 serve the same TMEM
    // lanes and split the work): S0 -> bf16 hi/lo A operand; X^T; gamma X_Q
    // and R
    {
        const int c = quad * 32 + lane;  // value column (TMEM lane)
        const int grp = warp >> 2;       // which half of each box / of the nodes
#pragma unroll 1
        for (int bx = 0; bx < 4; ++bx) {
            const int slot = bx & 1;
            if (!mbar_wait(&bars[BAR_S0 + slot], uint32_t(bx >> 1))) *sFlag = 1;
            const uint8_t* rowp = sm + L::S0S + slot * L::S0_BOX + c * 128;
            uint32_t wh[8], wl[8];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int j = 4 * grp + jj;  // 16-byte chunk of the row: 4 keys
                const float4 f = *reinterpret_cast<const float4*>(rowp + ((j ^ (c & 7)) << 4));
                split2(f.x, f.y, wh[2 * jj], wl[2 * jj]);
                split2(f.z, f.w, wh[2 * jj + 1], wl[2 * jj + 1]);
            }
            tmem_st8(lane_base + TA + bx * 16 + 8 * grp, wh);
            tmem_st8(lane_base + TA + 64 + bx * 16 + 8 * grp, wl);
            tmem_wait_st();
            tc_fence_before();
            __syncthreads();  // every thread has read (and stored) box bx
            if (tid == 128) {
                if (bx < 2) {
                    mbar_expect_tx(&bars[BAR_S0 + slot], L::S0_BOX);
                    tma_load_4d(sm + L::S0S + slot * L::S0_BOX, &tmS, &bars[BAR_S0 + slot], 32 * (bx + 2), 0, h,
                                b);
                }
                if (bx & 1) {
                    // X^T = S0 [Q_r; K_r]^T over the 64 keys of boxes bx - 1, bx
                    const int hv = bx >> 1;
                    if (hv == 0 && !mbar_wait(&bars[BAR_QK], 0)) *sFlag = 1;
                    tc_fence_after();
                    const uint32_t aQK = smem_u32(sQK);
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            const int ks = 4 * hv + k4;
                            const uint64_t db = sdesc_sw128(aQK + hv * 16384 + k4 * 32);
                            mma_bf16_ts(tmem + TX, tmem + TA + part * 64 + ks * 8, db, idesc_bf16(128, 128),
                                        (hv | part | k4) != 0);
                        }
                    if (hv == 1) mma_commit(&bars[BAR_X]);
                }
            }
        }
        if (!mbar_wait(&bars[BAR_X], 0)) *sFlag = 1;
        if (!mbar_wait(&bars[BAR_V], 0)) *sFlag = 1;
        tc_fence_after();
        const uint8_t* vt = sm + L::VT + (c >> 6) * L::V_TILE;
        const int cb = (c & 63) >> 3, cw = (c & 7) << 1;
#pragma unroll 1
        for (int nb = 32 * grp; nb < 32 * grp + 32; nb += 16) {
            uint32_t xq[16], xk[16];
            tmem_ld16(lane_base + TX + nb, xq);
            tmem_ld16(lane_base + TX + 64 + nb, xk);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int n = nb + e, i = n0 + n;
                if (i < T) {
                    const size_t ni = (size_t(b) * T + i) * H + h;
                    const float2 bg = sBG[n];
                    const float vv = __bfloat162float(
                        *reinterpret_cast<const __nv_bfloat16*>(vt + n * 128 + ((cb ^ (n & 7)) << 4) + cw));
                    ws.xq[ni * DV + c] = bg.y * __uint_as_float(xq[e]);
                    ws.rr[ni * DV + c] = bg.x * (vv - bg.y * __uint_as_float(xk[e]));
                }
            }
        }
    }
    // the staging area, V and the tensor-memory columns are free
    tc_fence_before();
    __syncthreads();

    // ---- phase 2: [Q_r; K_r] K_s^T for s = 0..r, then C and G row segments --
    if (tid == 0) {
        tc_fence_after();
        bool ok = !*sFlag;
        const uint32_t aQK = smem_u32(sQK), aKS = smem_u32(sm + L::KS);
        if (ok && r > 0) {
            mbar_expect_tx(&bars[BAR_KS], r * L::KS_TILE);
            for (int s = 0; s < r; ++s) {
                tma_load_4d(sm + L::KS + s * L::KS_TILE, &tmK, &bars[BAR_KS], 0, hk, TP * s, b);
                tma_load_4d(sm + L::KS + s * L::KS_TILE + 8192, &tmK, &bars[BAR_KS], 64, hk, TP * s, b);
            }
        }
        // the diagonal tile first (K_r is at hand), then the earlier ones
        for (int t = 0; t <= r; ++t) {
            const int s = (t == 0) ? r : t - 1;
            if (t == 1 && !mbar_wait(&bars[BAR_KS], 0)) {
                *sFlag = 1;
                ok = false;
            }
            if (!ok) break;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t da = sdesc_sw128(aQK + (ks >> 2) * 16384 + (ks & 3) * 32);
                const uint64_t db = (s == r) ? sdesc_sw128(aQK + (ks >> 2) * 16384 + 8192 + (ks & 3) * 32)
                                             : sdesc_sw128(aKS + s * L::KS_TILE + (ks >> 2) * 8192 + (ks & 3) * 32);
                mma_bf16_ss(tmem + TG + 64 * s, da, db, idesc_bf16(128, 64), ks != 0);
            }
        }
        mma_commit(&bars[BAR_AC]);
    }
    __syncwarp();
    if (!mbar_wait(&bars[BAR_AC], 0)) *sFlag = 1;
    tc_fence_after();
    {
        const int rho = tid & 127;           // TMEM lane: Q row rho, or K row rho - 64
        const bool qrow = rho < TP;
        const int e = rho & (TP - 1), i = n0 + e;
        const float li = sL[min(i, T - 1)];
        const float sc = qrow ? 1.f : sBG[e].x;
        float* dst = (qrow ? ws.cs : ws.gs) + ((size_t(b) * H + h) * T + min(i, T - 1)) * T;
        const bool vec = (T & 3) == 0;
        // warps w and w + 4 serve the same rows and take alternate tiles
        for (int s = warp >> 2; s <= r && !*sFlag; s += 2) {
            uint32_t m0 = sMask[e * 8 + 2 * s], m1 = sMask[e * 8 + 2 * s + 1];
            if (qrow && s == r) {  // C: i on its own path
                if (e < 32) m0 |= 1u << e;
                else m1 |= 1u << (e - 32);
            }
            const int jn = min(64, T - TP * s);  // columns inside the tree
            float* drow = dst + TP * s;
#pragma unroll 1
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t a[16];
                tmem_ld16(lane_base + TG + 64 * s + 16 * q4, a);
                tmem_wait_ld();
                if (i >= T) continue;
                float vals[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int jj = 16 * q4 + u;
                    const uint32_t bit = (jj < 32) ? ((m0 >> jj) & 1u) : ((m1 >> (jj - 32)) & 1u);
                    const int j = TP * s + jj;
                    vals[u] = bit ? sc * expf(li - sL[min(j, T - 1)]) * __uint_as_float(a[u]) : 0.f;
                }
                if (vec && 16 * q4 + 16 <= jn) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<float4*>(drow + 16 * q4 + 4 * q) =
                            make_float4(vals[4 * q], vals[4 * q + 1], vals[4 * q + 2], vals[4 * q + 3]);
                } else {
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        if (16 * q4 + u < jn) drow[16 * q4 + u] = vals[u];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *sFlag) {
        // a wait gave up: let the copies in flight land before leaving
        raise_err(ws.err, CANOPY_DEVERR_TIMEOUT);
        mbar_wait(&bars[BAR_QK], 0);
        if (r > 0) mbar_wait(&bars[BAR_KS], 0);  // (bounded; it gives up if the copies were never issued)
        for (int i = 0; i < 4; ++i) mbar_wait(&bars[BAR_S0 + (i & 1)], uint32_t(i >> 1));
        mbar_wait(&bars[BAR_V], 0);
    }
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace gtc

// ---------------------------------------------------------------------------
// Host side.

bool make_bf16_row_map(CUtensorMap* m, const void* base, int B, int T, int H);
bool make_state_map(CUtensorMap* m, const float* base, int B, int H);

cudaError_t launch_gram_tc(const void* q, const void* k, const void* v, const float* beta, const float* S0, int T,
                           int B, int H, int HK, const Ws& ws, cudaStream_t st) {
    CUtensorMap mq, mk, mv, ms;
    if (!make_bf16_row_map(&mq, q, B, T, HK) || !make_bf16_row_map(&mk, k, B, T, HK) ||
        !make_bf16_row_map(&mv, v, B, T, H) || !make_state_map(&ms, S0, B, H))
        return cudaErrorInvalidValue;
    const int smem = gtc::Smem::TOTAL + 1024;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(gtc::gram_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 grid((T + gtc::TP - 1) / gtc::TP, H, B);
    gtc::gram_tc_kernel<<<grid, gtc::NT, smem, st>>>(mq, mk, mv, ms, beta, T, H, HK, ws);
    return cudaGetLastError();
}

}  // namespace canopy
