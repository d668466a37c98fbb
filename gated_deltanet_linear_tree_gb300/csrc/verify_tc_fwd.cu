// Closed-form tree verify on tcgen05 tensor cores, forward-substitution solve,
// one 64-node block (T <= 64), bf16 q/k/v, fp32 S0, fp32 accumulation.
//
// Method: canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed
// form" (Bole's Theorem 1):
//     (I + G) U = R,  R = diag(beta) (V - diag(gamma) K S0^T),
//     O = diag(gamma) Q S0^T + C U,
// carried by the inverse W = (I + G)^-1 (ancestor sparsity) and M = C W:
//     U = W R,   O = diag(gamma) Q S0^T + M R.
//
// One CTA (256 threads) owns one (stream b, head h).  Its two warp groups
// work concurrently:
//   solve warps 0-3:  tree prep (each node walks its parent chain: path
//       bitmask, depth, cumulative log2 gate); the Gram block AC = [Q;K] K^T
//       on tcgen05; C and G rows with the decay 2^(l2_i - l2_j) on the
//       root-path entries, compacted to path positions; W and M rows by
//       right-looking substitution along each node's root path (rows are
//       independent: W (I + G) = I, M (I + G) = C); [M; W] to shared memory
//       as bf16 hi + lo (the B operand of the output product).
//   state warps 4-7:  S0 rows -> bf16 hi + lo in tensor memory (the A
//       operand); X^T = S0 [Q;K]^T on tcgen05 (value columns on the TMEM
//       lanes, nodes on the columns); R^T = beta (V - gamma X_K)^T as bf16
//       hi + lo into tensor memory; the X_Q columns scaled by gamma.
// Then Y^T = [gamma X_Q^T | 0] + R^T [M; W]^T by three bf16 products
// (hi*hi + hi*lo + lo*hi, ~16 mantissa bits each side), and each warp stores
// 32 value columns of o (warps 0-3) or U (warps 4-7) for every node.
// Decay ratios are only ever 2^(l2_i - l2_j) with j on i's root path, so they
// lie in (0, 1] and never overflow ("Hard constraints", log-space gates).
#include "common.cuh"

namespace canopy {

namespace tcf {

constexpr int DK = 128;
constexpr int DV = 128;
constexpr int TP = 64;    // nodes per block
constexpr int NT = 256;   // threads per CTA
constexpr int XS = 68;    // row stride (floats) of the per-row work vectors and of Gp
constexpr uint32_t kTmemCols = 256;
// tensor-memory columns
constexpr uint32_t TA = 0;      // S0 as A: hi [0,64), lo [64,128); later R^T: hi [0,32), lo [32,64)
constexpr uint32_t TD = 128;    // AC [128,192) first; then X^T / Y^T [128,256): o part [128,192), U part [192,256)

struct Smem {
    static constexpr int QK = 0;                 // [Q;K] bf16, 2 atoms x 128 rows x 128 B; later [M;W] hi/lo
    static constexpr int BH = 0;                 // [M;W] bf16 hi: 128 rows x 128 B
    static constexpr int BL = 16384;             // [M;W] bf16 lo
    static constexpr int VT = 32768;             // V bf16: 2 tiles [64 nodes][64 cols], 128-byte swizzle
    static constexpr int V_TILE = 64 * 128;
    static constexpr int XV = VT + 2 * V_TILE;   // per-row work vectors fp32 [128][XS]
    static constexpr int GP = XV + 128 * XS * 4; // Gp fp32 [64][XS]: G rows by path position
    static constexpr int PAR = GP + TP * XS * 4; // int[64] parent
    static constexpr int LEN = PAR + 256;        // int[64] path length
    static constexpr int L2 = LEN + 256;         // float[64] log2 gate, then cumulative
    static constexpr int GAM = L2 + 256;         // float[64] gamma
    static constexpr int BETA = GAM + 256;       // float[64]
    static constexpr int MASK = BETA + 256;      // u64[64] path(i), i included
    static constexpr int BAR = MASK + 512;       // u64[8]
    static constexpr int TMEMSLOT = BAR + 64;    // u32
    static constexpr int FLAG = TMEMSLOT + 4;    // int
    static constexpr int PLIST = FLAG + 12;      // u8[64][64] path(i) from the root down
    static constexpr int TOTAL = PLIST + TP * TP;
    static_assert(XV % 16 == 0 && GP % 16 == 0, "align");
};

enum { BAR_QK = 0, BAR_V, BAR_PREP, BAR_AC, BAR_ACC, BAR_X, BAR_Y, NBAR };

struct Params {
    const float* g;
    const float* beta;
    const float* S0;
    const int32_t* parent;
    void* o;
    float* U;
    float* l;
    int32_t* depth;
    uint32_t* mask;
    int32_t* err;
    int B, T, H, W, o_bf16;
};

__device__ inline uint32_t pack_bf16(float lo_half, float hi_half) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo_half, hi_half);
    return *reinterpret_cast<const uint32_t*>(&p);
}

// x -> bf16 hi (round to nearest) and bf16 lo = bf16(x - hi).
__device__ inline void split_bf16(float x, float& hi, float& lo) {
    hi = __bfloat162float(__float2bfloat16_rn(x));
    lo = x - hi;
}

__device__ inline void wait_or_flag(uint64_t* bar, int* sFlag) {
    if (!mbar_wait(bar, 0)) *sFlag = 1;
}

__global__ void __launch_bounds__(NT, 2)
    verify_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, Params p) {
    using L = Smem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* sPar = reinterpret_cast<int*>(sm + L::PAR);
    int* sLen = reinterpret_cast<int*>(sm + L::LEN);
    float* sL2 = reinterpret_cast<float*>(sm + L::L2);
    float* sGam = reinterpret_cast<float*>(sm + L::GAM);
    float* sBeta = reinterpret_cast<float*>(sm + L::BETA);
    uint64_t* sMask = reinterpret_cast<uint64_t*>(sm + L::MASK);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + L::TMEMSLOT);
    int* sFlag = reinterpret_cast<int*>(sm + L::FLAG);
    uint8_t* sPath = sm + L::PLIST;
    float* sX = reinterpret_cast<float*>(sm + L::XV);
    float* sGp = reinterpret_cast<float*>(sm + L::GP);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3;                  // TMEM lane quadrant of this warp
    const bool solve = warp < 4;
    const int h = blockIdx.x, b = blockIdx.y;
    const int T = p.T, H = p.H;
    const float* S0 = p.S0 + (size_t(b) * H + h) * DV * DK;

    uint8_t* sQK = sm + L::QK;
    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        *sFlag = 0;
        // Q and K first: the solve path waits on them
        mbar_expect_tx(&bars[BAR_QK], 4 * 64 * 64 * 2);
        tma_load_4d(sQK + 0, &tmQ, &bars[BAR_QK], 0, h, 0, b);
        tma_load_4d(sQK + 16384, &tmQ, &bars[BAR_QK], 64, h, 0, b);
        tma_load_4d(sQK + 8192, &tmK, &bars[BAR_QK], 0, h, 0, b);
        tma_load_4d(sQK + 24576, &tmK, &bars[BAR_QK], 64, h, 0, b);
    }
    if (warp == 0) {
        tmem_alloc(sTmem, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    // Parents and gates (threads 0..63); padded nodes: no path, beta 0, gamma 1.
    if (tid < TP) {
        const int i = tid;
        int par = -1, bad = 0;
        float a = 1.f, be = 0.f;
        if (i < T) {
            par = p.parent[size_t(b) * T + i];
            a = p.g[(size_t(b) * T + i) * H + h];
            be = p.beta[(size_t(b) * T + i) * H + h];
            if (!((i == 0) ? (par == -1) : (par >= 0 && par < i))) {
                bad |= CANOPY_DEVERR_TREE;
                par = (i == 0) ? -1 : 0;
            }
            if (!gate_ok(a, be)) {
                bad |= CANOPY_DEVERR_GATE;
                a = 1.f;
                be = 0.f;
            }
        }
        if (bad) raise_err(p.err, bad);
        sPar[i] = par;
        sL2[i] = log2f(a);
        sBeta[i] = be;
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16);


    if (solve) {
        // ---- tree prep: node i walks its (sanitised) parent chain ----------
        float myl2 = 0.f;
        if (tid < TP) {
            const int i = tid;
            uint64_t m = 0;
            int n = 0;
            if (i < T) {
                float s = 0.f;
                for (int j = i; j >= 0; j = sPar[j]) {
                    m |= 1ull << j;
                    s += sL2[j];
                    ++n;
                }
                myl2 = s;
            }
            sMask[i] = m;
            sLen[i] = n;
        }
        group_sync(1, 128);
        if (tid < TP) {
            const int i = tid;
            sL2[i] = myl2;  // every walk has read the per-node gates by now
            sGam[i] = exp2f(myl2);
            if (i < T) {
                int d = 0;
                for (uint64_t bits = sMask[i]; bits; bits &= bits - 1)
                    sPath[i * TP + d++] = uint8_t(__ffsll(static_cast<long long>(bits)) - 1);
            }
        }
        group_sync(1, 128);
        if (tid == 0) mbar_arrive(&bars[BAR_PREP]);  // gamma is ready for the state warps

        // ---- C and G rows from AC (lane r: Q row r, or K row r - 64) ----------
        const int r = tid;                     // 0..127: TMEM lane of this thread
        const bool qrow = r < TP;
        const int i = r & (TP - 1);
        float* xr = sX + r * XS;               // this row's work vector
        wait_or_flag(&bars[BAR_AC], sFlag);
        tc_fence_after();
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
            uint32_t a[32];
            tmem_ld16(lane_base + TD + hc * 32, *reinterpret_cast<uint32_t(*)[16]>(a));
            tmem_ld16(lane_base + TD + hc * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(a + 16));
            tmem_wait_ld();
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4)
                *reinterpret_cast<float4*>(xr + hc * 32 + 4 * j4) =
                    make_float4(__uint_as_float(a[4 * j4]), __uint_as_float(a[4 * j4 + 1]),
                                __uint_as_float(a[4 * j4 + 2]), __uint_as_float(a[4 * j4 + 3]));
        }
        tc_fence_before();
        group_sync(1, 128);
        if (tid == 0) mbar_arrive(&bars[BAR_ACC]);  // the AC columns may be overwritten

        const int n = (i < T) ? sLen[i] : 0;
        const uint8_t* pl = sPath + i * TP;
        const float li = sL2[i];
        // C row (Q lanes) or G row (K lanes, strict ancestors, scaled by beta)
        // by path position, four positions per batch (loads before stores;
        // the C row is compacted in place: position d <= node id j, and a
        // batch writes only positions below every later read).
        {
            const int cnt = qrow ? n : n - 1;
            float* dst = qrow ? xr : sGp + i * XS;
            const float sc = qrow ? 1.f : sBeta[i];
            for (int d0 = 0; d0 < cnt; d0 += 4) {
                float v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int j = pl[min(d0 + u, cnt - 1)];
                    v[u] = sc * exp2f(li - sL2[j]) * xr[j];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (d0 + u < cnt) dst[d0 + u] = v[u];
            }
            if (!qrow && n > 0) {
                // Gp row zero-padded by 4; the work vector becomes e_(n-1)
#pragma unroll
                for (int z = 0; z < 4; ++z) dst[n - 1 + z] = 0.f;
                for (int d = 0; d < n; ++d) xr[d] = (d == n - 1) ? 1.f : 0.f;
            }
        }
        group_sync(1, 128);

        // ---- W and M rows: right-looking substitution along path(i) ----------
        // x_d -= x_e Gp[pl[e]][d] for e = n-1 .. 1 and d < e; Gp rows are
        // zero beyond their length, so whole float4 groups are safe.
        for (int e = n - 1; e >= 1; --e) {
            const float xe = xr[e];
            const float* gr = sGp + pl[e] * XS;
            for (int d = 0; d < e; d += 4) {
                float4 x4 = *reinterpret_cast<const float4*>(xr + d);
                const float4 g4 = *reinterpret_cast<const float4*>(gr + d);
                x4.x -= xe * g4.x;
                x4.y -= xe * g4.y;
                x4.z -= xe * g4.z;
                x4.w -= xe * g4.w;
                *reinterpret_cast<float4*>(xr + d) = x4;
            }
        }

        // ---- [M; W] row r -> B operand (K-major bf16, 128-byte swizzle) ---------
        wait_or_flag(&bars[BAR_X], sFlag);  // the [Q;K] tile is no longer read
        {
            uint8_t* bh = sm + L::BH + r * 128;
            uint8_t* bl = sm + L::BL + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                *reinterpret_cast<uint4*>(bh + (c << 4)) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(bl + (c << 4)) = make_uint4(0, 0, 0, 0);
            }
            for (int d = 0; d < n; ++d) {
                const int j = pl[d];
                float hi, lo;
                split_bf16(xr[d], hi, lo);
                const int off = ((((j >> 3) ^ (r & 7))) << 4) + ((j & 7) << 1);
                *reinterpret_cast<__nv_bfloat16*>(bh + off) = __float2bfloat16_rn(hi);
                *reinterpret_cast<__nv_bfloat16*>(bl + off) = __float2bfloat16_rn(lo);
            }
        }
        fence_proxy_async_smem();
        // tree outputs for the commit: l (natural log), depth, strict-ancestor mask
        if (tid < TP && tid < T) {
            p.l[(size_t(b) * T + tid) * H + h] = sL2[tid] * 0.69314718055994531f;
            if (h == 0) {
                p.depth[size_t(b) * T + tid] = sLen[tid] - 1;
                const uint64_t strict = sMask[tid] & ~(1ull << tid);
                for (int w = 0; w < p.W; ++w)
                    p.mask[(size_t(b) * T + tid) * p.W + w] = uint32_t(strict >> (32 * w));
            }
        }
    } else {
        // ---- state warps: S0 rows -> bf16 hi/lo A operand in tensor memory ----
        // AC = [Q;K] K^T (M = 128, N = 64) as soon as Q and K have landed;
        // then V and S0 are requested (Q and K come first from HBM).
        const int c = quad * 32 + lane;  // value column of this thread in the R and store phases
        if (tid == 128) {
            if (mbar_wait(&bars[BAR_QK], 0)) {
                tc_fence_after();
                const uint32_t aQK = smem_u32(sQK);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t da = sdesc_sw128(aQK + (ks >> 2) * 16384 + (ks & 3) * 32);
                    const uint64_t db = sdesc_sw128(aQK + (ks >> 2) * 16384 + 8192 + (ks & 3) * 32);
                    mma_bf16_ss(tmem + TD, da, db, idesc_bf16(128, 64), ks != 0);
                }
            } else {
                *sFlag = 1;
            }
            mma_commit(&bars[BAR_AC]);
            mbar_expect_tx(&bars[BAR_V], 2 * L::V_TILE);
            tma_load_4d(sm + L::VT, &tmV, &bars[BAR_V], 0, h, 0, b);
            tma_load_4d(sm + L::VT + L::V_TILE, &tmV, &bars[BAR_V], 64, h, 0, b);
        }
        __syncwarp();
        // S0 row (32 quad + 16 half + lane/4 [+ 8]) -> tensor-memory lane of the
        // same index; each group of four threads reads 64 contiguous bytes of
        // a row (16 dk values = 8 columns of bf16 pairs).
        {
            const int rsub = lane >> 2, csub = lane & 3;
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                const int row0 = quad * 32 + hf * 16 + rsub;
                const float4* r0p = reinterpret_cast<const float4*>(S0 + size_t(row0) * DK) + csub;
                const float4* r1p = reinterpret_cast<const float4*>(S0 + size_t(row0 + 8) * DK) + csub;
                const uint32_t taddr = tmem + (uint32_t(quad * 32 + hf * 16) << 16);
#pragma unroll 2
                for (int grp = 0; grp < 2; ++grp) {      // 32 columns = 64 dk values per group
                    float4 f0[4], f1[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        f0[k] = r0p[(grp * 4 + k) * 4];
                        f1[k] = r1p[(grp * 4 + k) * 4];
                    }
                    uint32_t wh[16], wl[16];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float h0, l0, h1, l1, h2, l2, h3, l3;
                        split_bf16(f0[k].x, h0, l0);
                        split_bf16(f0[k].y, h1, l1);
                        split_bf16(f0[k].z, h2, l2);
                        split_bf16(f0[k].w, h3, l3);
                        wh[4 * k] = pack_bf16(h0, h1);
                        wh[4 * k + 1] = pack_bf16(h2, h3);
                        wl[4 * k] = pack_bf16(l0, l1);
                        wl[4 * k + 1] = pack_bf16(l2, l3);
                        split_bf16(f1[k].x, h0, l0);
                        split_bf16(f1[k].y, h1, l1);
                        split_bf16(f1[k].z, h2, l2);
                        split_bf16(f1[k].w, h3, l3);
                        wh[4 * k + 2] = pack_bf16(h0, h1);
                        wh[4 * k + 3] = pack_bf16(h2, h3);
                        wl[4 * k + 2] = pack_bf16(l0, l1);
                        wl[4 * k + 3] = pack_bf16(l2, l3);
                    }
                    tmem_st_16x256b_x4(taddr + TA + grp * 32, wh);
                    tmem_st_16x256b_x4(taddr + TA + 64 + grp * 32, wl);
                }
            }
        }
        tmem_wait_st();
        tc_fence_before();
        group_sync(2, 128);
        if (tid == 128) {
            // X^T = S0 [Q;K]^T (M = 128 value rows, N = 128 nodes) once the
            // AC columns have been read out
            if (!mbar_wait(&bars[BAR_ACC], 0)) *sFlag = 1;
            tc_fence_after();
            const uint32_t aQK = smem_u32(sQK);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t db = sdesc_sw128(aQK + (ks >> 2) * 16384 + (ks & 3) * 32);
                    mma_bf16_ts(tmem + TD, tmem + TA + part * 64 + ks * 8, db, idesc_bf16(128, 128),
                                (part | ks) != 0);
                }
            mma_commit(&bars[BAR_X]);
        }
        __syncwarp();

        // ---- R^T = beta (V - gamma X_K)^T and gamma X_Q^T ---------------------
        wait_or_flag(&bars[BAR_X], sFlag);
        wait_or_flag(&bars[BAR_V], sFlag);
        wait_or_flag(&bars[BAR_PREP], sFlag);
        tc_fence_after();
        {
            const uint8_t* vt = sm + L::VT + (c >> 6) * L::V_TILE;
            const int cb = ((c & 63) >> 3), cw = (c & 7) << 1;
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t xk[16];
                tmem_ld16(lane_base + TD + 64 + blk * 16, xk);
                tmem_wait_ld();
                uint32_t wh[8], wl[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float rv[2];
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        const int i = blk * 16 + 2 * e + s;
                        const float vv = __bfloat162float(
                            *reinterpret_cast<const __nv_bfloat16*>(vt + i * 128 + ((cb ^ (i & 7)) << 4) + cw));
                        rv[s] = (i < T) ? sBeta[i] * (vv - sGam[i] * __uint_as_float(xk[2 * e + s])) : 0.f;
                    }
                    float h0, l0, h1, l1;
                    split_bf16(rv[0], h0, l0);
                    split_bf16(rv[1], h1, l1);
                    wh[e] = pack_bf16(h0, h1);
                    wl[e] = pack_bf16(l0, l1);
                }
                tmem_st8(lane_base + TA + blk * 8, wh);
                tmem_st8(lane_base + TA + 32 + blk * 8, wl);
            }
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t xq[16];
                tmem_ld16(lane_base + TD + blk * 16, xq);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) xq[e] = __float_as_uint(sGam[blk * 16 + e] * __uint_as_float(xq[e]));
                tmem_st16(lane_base + TD + blk * 16, xq);
            }
            tmem_wait_st();
        }
        tc_fence_before();
    }
    __syncthreads();

    // ---- Y^T = [gamma X_Q^T | 0] + R^T [M; W]^T (bf16 x3) -------------------------
    if (tid == 128) {
        tc_fence_after();
        const uint32_t bH = smem_u32(sm + L::BH), bL = smem_u32(sm + L::BL);
#pragma unroll 1
        for (int part = 0; part < 2; ++part) {        // 0: o (M rows), 1: U (W rows)
            const uint32_t d = tmem + TD + part * 64;
            const uint32_t rowoff = part * 64 * 128;
#pragma unroll 1
            for (int pass = 0; pass < 3; ++pass) {    // hi*hi, hi*lo, lo*hi
                const uint32_t acol = TA + (pass == 2 ? 32 : 0);
                const uint32_t bb = (pass == 1 ? bL : bH) + rowoff;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ts(d, tmem + acol + ks * 8, sdesc_sw128(bb + ks * 32), idesc_bf16(128, 64),
                                (part == 0) || pass != 0 || ks != 0);
            }
        }
        mma_commit(&bars[BAR_Y]);
    }
    __syncwarp();
    wait_or_flag(&bars[BAR_Y], sFlag);
    tc_fence_after();

    // ---- store: warps 0-3 o, warps 4-7 U; lane = value column --------------------
    {
        const int c = quad * 32 + lane;
        const uint32_t col0 = TD + (solve ? 0 : 64);
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
            uint32_t y[16];
            tmem_ld16(lane_base + col0 + blk * 16, y);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int i = blk * 16 + e;
                if (i < T) {
                    const size_t off = ((size_t(b) * T + i) * H + h) * DV + c;
                    const float yv = __uint_as_float(y[e]);
                    if (!solve)
                        p.U[off] = yv;
                    else if (p.o_bf16)
                        static_cast<__nv_bfloat16*>(p.o)[off] = __float2bfloat16_rn(yv);
                    else
                        static_cast<float*>(p.o)[off] = yv;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (tid == 128 && *sFlag) {
        // a wait gave up: let the copies in flight land before leaving
        raise_err(p.err, CANOPY_DEVERR_TIMEOUT);
        mbar_wait(&bars[BAR_QK], 0);
        mbar_wait(&bars[BAR_V], 0);
    }
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace tcf

// ---------------------------------------------------------------------------
// Host side.

bool make_bf16_row_map(CUtensorMap* m, const void* base, int B, int T, int H);

cudaError_t launch_verify_tc_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                 const float* S0, const int32_t* parent, int T, int B, int H, void* o, int o_bf16,
                                 const Ws& ws, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    if (!make_bf16_row_map(&mq, q, B, T, H) || !make_bf16_row_map(&mk, k, B, T, H) ||
        !make_bf16_row_map(&mv, v, B, T, H))
        return cudaErrorInvalidValue;
    tcf::Params prm;
    prm.g = g;
    prm.beta = beta;
    prm.S0 = S0;
    prm.parent = parent;
    prm.o = o;
    prm.U = ws.U;
    prm.l = ws.l;
    prm.depth = ws.depth;
    prm.mask = ws.mask;
    prm.err = ws.err;
    prm.B = B;
    prm.T = T;
    prm.H = H;
    prm.W = ws.W;
    prm.o_bf16 = o_bf16;
    const int smem = tcf::Smem::TOTAL + 1024;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(tcf::verify_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    tcf::verify_fwd_kernel<<<dim3(H, B), tcf::NT, smem, st>>>(mq, mk, mv, prm);
    return cudaGetLastError();
}

}  // namespace canopy
