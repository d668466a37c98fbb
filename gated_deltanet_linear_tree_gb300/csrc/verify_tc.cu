// Closed-form tree verify with the finite Neumann series solve, on tcgen05
// tensor cores (bf16 q/k/v, fp32 S0, fp32 accumulation in tensor memory), one
// 64-node block (T <= 64).  The forward-substitution kernel is the default
// path; this variant is the solve of the canopy page's "Design decisions"
// (Bole's solve), kept selectable and checked against the same oracle.
//
// Method: canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed
// form" (Bole's Theorem 1):
//     (I + G) U = R,  R = diag(beta) (V - diag(gamma) K S0^T),
//     O = diag(gamma) Q S0^T + C U.
// G is strictly lower triangular on the ancestor pattern, so (-G)^m = 0 once
// m exceeds the tree depth d and W = (I + G)^-1 = sum_{m=0..d} (-G)^m exactly.
// With M = C W:  U = W R,  O = diag(gamma) Q S0^T + M R.
// One CTA (256 threads) owns one (stream b, head h) and all 128 value columns:
//   1. tree prep: parent -> path bitmask, depth, l_i = sum log2 alpha, by
//      pointer jumping;
//   2. AC = [Q;K] K^T and X = [Q;K] S0^T on tcgen05 in one commit (M = 128:
//      Q rows then K rows); S0 is split into bf16 hi + lo in shared memory so
//      X keeps ~16 mantissa bits of fp32; C_ij = 2^(l2_i - l2_j) q_i.k_j and
//      G_ij = beta_i 2^(l2_i - l2_j) k_i.k_j on the root-path entries go to
//      shared memory;
//   3. W by d rounds P_m = -G P_(m-1) on tcgen05 (G as the tf32 hi + lo A
//      operand in tensor memory, P^T as the B operand in shared memory, three
//      products per round), then M = C W on the CUDA cores;
//   4. [M; W] is written to tensor memory as tf32 hi + lo parts;
//   5. R = beta (V - gamma X_K) goes to shared memory as tf32 hi + lo; the
//      X_Q rows are scaled by gamma and the X_K rows zeroed in place; then
//      X += [M; W] R by three tf32 MMAs (hi*hi + hi*lo + lo*hi), which keeps
//      fp32 accuracy: rows 0..63 become o, rows 64..127 become U.
// Decay ratios are only ever 2^(l2_i - l2_j) with j on i's root path, so they
// lie in (0, 1] and never overflow ("Hard constraints", log-space gates).
// This file also holds the tensor-map encoders both tensor-core kernels use.
#include "common.cuh"

namespace canopy {

namespace tc {

constexpr int DK = 128;
constexpr int DV = 128;
constexpr int TP = 64;       // nodes per block
constexpr int RS = 65;       // padded row stride (floats) of the T x T tables
constexpr int NT = 256;      // threads per CTA
// X [0,128), A hi [128,192), A lo [192,256), the products G P at [256,320)
constexpr uint32_t kTmemColsNeu = 512;
constexpr int YC = 256;
constexpr int XC = 0, AH = 128, AL = 192;

struct Smem {
    // phase 1: Q/K and S0 hi/lo (until the first products complete)
    static constexpr int QK = 0;                 // [Q;K] bf16: 2 atoms x 128 rows x 128 B
    static constexpr int S = 32768;              // S0: 2 planes x 2 atoms x 128 rows x 128 B
    static constexpr int S_ATOM = 128 * 128;
    static constexpr int S_PLANE = 2 * S_ATOM;
    static constexpr int P1_END = S + 2 * S_PLANE;
    // phase 2: the T x T tables (over phase 1) and V (loaded by TMA once
    // phase 1 is done)
    static constexpr int CT = 0;                 // C fp32 [64][RS]
    static constexpr int GT = CT + TP * RS * 4;  // G
    static constexpr int WT = GT + TP * RS * 4;  // W
    static constexpr int MT = WT + TP * RS * 4;  // M
    static constexpr int VT = 67584;             // V bf16: 2 tiles [64 nodes][64 cols], 128-byte swizzle
    static constexpr int V_TILE = 64 * 128;
    static constexpr int P2_END = VT + 2 * V_TILE;
    // phase 3: R^T hi/lo as the K-major tf32 B operand [128 cols][64 nodes]
    static constexpr int RH = 0;
    static constexpr int RL = 32768;
    static constexpr int R_ATOM = 128 * 128;     // 32 nodes x 128 rows
    // small arrays
    static constexpr int SMALL = 98304;
    static constexpr int PAR = SMALL;            // int[64]   jump pointer
    static constexpr int LEN = PAR + 256;        // int[64]   path length
    static constexpr int L2 = LEN + 256;         // float[64] cumulative log2 gate
    static constexpr int GAM = L2 + 256;         // float[64] gamma = 2^l2
    static constexpr int BETA = GAM + 256;       // float[64]
    static constexpr int MASK = BETA + 256;      // u64[64]   path(i) incl. i
    static constexpr int BAR = MASK + 512;       // u64[3]
    static constexpr int TMEMSLOT = BAR + 24;    // u32
    static constexpr int FLAG = TMEMSLOT + 4;    // int
    static constexpr int DMAX = FLAG + 4;        // int: tree depth
    static constexpr int PLIST = DMAX + 4;       // u8[64][64]: path(i) from the root down
    static constexpr int TOTAL = PLIST + TP * TP;
    // Neumann: P^T hi/lo operand [64 rows][64] tf32 (after the small arrays)
    static constexpr int PH = (TOTAL + 1023) & ~1023;
    static constexpr int PL = PH + 16384;
    static constexpr int P_ATOM = 64 * 128;
    static constexpr int TOTAL_NEU = PL + 16384;
    static_assert(P1_END <= SMALL && MT + TP * RS * 4 <= VT && P2_END <= SMALL && RL + 2 * R_ATOM <= VT,
                  "layout");
};

struct Params {
    const __nv_bfloat16* v;
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
    int HK;       // key heads: value head h reads q and k of key head h / (H / HK)
    float scale;  // factor on q (applied to o)
};

__device__ inline float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ inline float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// tf32 hi/lo split for the three-product scheme: hi keeps the top 10
// mantissa bits (exact in tf32), lo = x - hi is exact in fp32; the tensor core
// reads lo to 10 bits, so hi + lo carries x to within 2^-20 |x|.
__device__ inline void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
    hi = __float_as_uint(x) & 0xFFFFE000u;
    lo = __float_as_uint(x - __uint_as_float(hi));
}

// Byte offset of element (row n, K index k) of a K-major tf32 operand in the
// 128-byte swizzle layout with `rows` rows per 32-wide K atom.
__device__ inline int kmajor_tf32_off(int n, int k, int rows) {
    return (k >> 5) * (rows * 128) + n * 128 + ((((k & 31) >> 2) ^ (n & 7)) << 4) + ((k & 3) << 2);
}

// The k-th (0-based) set bit of a 64-bit mask.
__device__ inline int nth_bit(uint64_t m, int k) {
    const uint32_t lo = uint32_t(m), hi = uint32_t(m >> 32);
    const int c = __popc(lo);
    return (k < c) ? int(__fns(lo, 0, k + 1)) : 32 + int(__fns(hi, 0, k - c + 1));
}

// Bounded wait on an mbarrier phase by warp 0; a timeout is recorded in sFlag.
__device__ inline void warp0_wait(uint64_t* bar, uint32_t parity, int* sFlag) {
    const bool ok = mbar_wait(bar, parity);
    if (!ok && (threadIdx.x & 31) == 0) *sFlag = 1;
}

__global__ void __launch_bounds__(NT, 2)
    verify_neumann_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, Params p) {
    using L = Smem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    int* sPtr = reinterpret_cast<int*>(sm + L::PAR);
    int* sLen = reinterpret_cast<int*>(sm + L::LEN);
    float* sL2 = reinterpret_cast<float*>(sm + L::L2);
    float* sGam = reinterpret_cast<float*>(sm + L::GAM);
    float* sBeta = reinterpret_cast<float*>(sm + L::BETA);
    uint64_t* sMask = reinterpret_cast<uint64_t*>(sm + L::MASK);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + L::TMEMSLOT);
    int* sFlag = reinterpret_cast<int*>(sm + L::FLAG);
    int* sDmax = reinterpret_cast<int*>(sm + L::DMAX);
    uint8_t* sPath = sm + L::PLIST;
    float* sC = reinterpret_cast<float*>(sm + L::CT);
    float* sG = reinterpret_cast<float*>(sm + L::GT);
    float* sW = reinterpret_cast<float*>(sm + L::WT);
    float* sM = reinterpret_cast<float*>(sm + L::MT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;      // TMEM lane quadrant, column half
    const int row = quad * 32 + lane;                 // TMEM lane: 0..63 Q rows, 64..127 K rows
    const int h = blockIdx.x, b = blockIdx.y;
    const int T = p.T, H = p.H;
    uint32_t mma_phase = 0;
    bool v_issued = false;

    if (tid == 0) {
        mbar_init(&bars[0], 1);  // Q/K
        mbar_init(&bars[1], 1);  // MMA completions
        mbar_init(&bars[2], 1);  // V
        fence_mbar_init();
        *sFlag = 0;
        *sDmax = 0;
    }
    if (warp == 0) {
        tmem_alloc(sTmem, kTmemColsNeu);
        tmem_relinquish();
        tc_fence_before();
    }

    // S0 (128 rows x 128 fp32 = 64 KiB, contiguous): 16-byte coalesced loads
    // issued first; the values are converted once the tables are done.
    float4 s0r[16];
    {
        const float4* src = reinterpret_cast<const float4*>(p.S0 + (size_t(b) * H + h) * DV * DK);
#pragma unroll
        for (int u = 0; u < 16; ++u) s0r[u] = __ldg(src + u * NT + tid);
    }
    // Parents and gates; padded nodes get no path, beta = 0 and gamma = 1.
    int bad = 0;
    if (tid < TP) {
        const int i = tid;
        int par = -1;
        float a = 1.f, be = 0.f;
        if (i < T) {
            par = p.parent[size_t(b) * T + i];
            a = p.g[(size_t(b) * T + i) * H + h];
            be = p.beta[(size_t(b) * T + i) * H + h];
            const bool ok_par = (i == 0) ? (par == -1) : (par >= 0 && par < i);
            if (!ok_par) {
                bad |= CANOPY_DEVERR_TREE;
                par = (i == 0) ? -1 : 0;
            }
            if (!gate_ok(a, be)) {
                bad |= CANOPY_DEVERR_GATE;
                a = 1.f;
                be = 0.f;
            }
        }
        sPtr[i] = par;
        sL2[i] = (i < T) ? log2f(a) : 0.f;
        sBeta[i] = be;
    }
    if (bad) raise_err(p.err, bad);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16);

    uint8_t* sQK = sm + L::QK;
    if (tid == 0) {
        mbar_expect_tx(&bars[0], 4 * 64 * 64 * 2);
        const int hk = h / (H / p.HK);
        tma_load_4d(sQK + 0, &tmQ, &bars[0], 0, hk, 0, b);
        tma_load_4d(sQK + 16384, &tmQ, &bars[0], 64, hk, 0, b);
        tma_load_4d(sQK + 8192, &tmK, &bars[0], 0, hk, 0, b);
        tma_load_4d(sQK + 24576, &tmK, &bars[0], 64, hk, 0, b);
    }

    // Tree prep (threads 0..63 own nodes; the whole CTA takes the barriers).
    jump_paths<1>(TP, sPtr, sLen, sL2, sMask);
    if (tid < TP) {
        const int i = tid;
        if (i >= T) sMask[i] = 0ull;  // padded nodes: empty path
        sGam[i] = exp2f(sL2[i]);
        if (i < T) {
            atomicMax(sDmax, sLen[i] - 1);
            // root path of i as a list of node ids, root first
            int d = 0;
            for (uint64_t bits = sMask[i]; bits; bits &= bits - 1)
                sPath[i * TP + d++] = uint8_t(__ffsll(static_cast<long long>(bits)) - 1);
            p.l[(size_t(b) * T + i) * H + h] = sL2[i] * 0.69314718055994531f;
            if (h == 0) {
                p.depth[size_t(b) * T + i] = sLen[i] - 1;
                const uint64_t strict = sMask[i] & ~(1ull << i);
                for (int w = 0; w < p.W; ++w)
                    p.mask[(size_t(b) * T + i) * p.W + w] = uint32_t(strict >> (32 * w));
            }
        }
    }
    __syncthreads();

    // S0 -> bf16 hi and lo planes (K-major, 128-byte swizzle), while the
    // tree prep is done.
    {
        uint8_t* sS = sm + L::S;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int f = u * NT + tid;
            const int r = f >> 5, c4 = f & 31;
            const int atom = c4 >> 4, chunk = (c4 & 15) >> 1;
            const int off = atom * L::S_ATOM + r * 128 + ((chunk ^ (r & 7)) << 4) + ((c4 & 1) << 3);
            const __nv_bfloat162 h01 = __floats2bfloat162_rn(s0r[u].x, s0r[u].y);
            const __nv_bfloat162 h23 = __floats2bfloat162_rn(s0r[u].z, s0r[u].w);
            const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
            const __nv_bfloat162 l01 = __floats2bfloat162_rn(s0r[u].x - f01.x, s0r[u].y - f01.y);
            const __nv_bfloat162 l23 = __floats2bfloat162_rn(s0r[u].z - f23.x, s0r[u].w - f23.y);
            *reinterpret_cast<uint2*>(sS + off) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
            *reinterpret_cast<uint2*>(sS + L::S_PLANE + off) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&l01), *reinterpret_cast<const uint32_t*>(&l23));
        }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // AC = [Q;K] K^T into the A-hi columns (rewritten later with [M; W]) and
    // X = [Q;K] S0^T, one commit.
    if (warp == 0) {
        const bool ok = mbar_wait(&bars[0], 0);
        if (lane == 0) {
            if (!ok) {
                *sFlag = 1;
            } else {
                tc_fence_after();
                const uint32_t aQK = smem_u32(sQK);
                const uint32_t aS = smem_u32(sm + L::S);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t da = sdesc_sw128(aQK + (ks >> 2) * 16384 + (ks & 3) * 32);
                    const uint64_t db = sdesc_sw128(aQK + (ks >> 2) * 16384 + 8192 + (ks & 3) * 32);
                    mma_bf16_ss(tmem + AH, da, db, idesc_bf16(128, 64), ks != 0);
                }
                // X = [Q;K] (S0hi + S0lo)^T, N = 128
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t da = sdesc_sw128(aQK + (ks >> 2) * 16384 + (ks & 3) * 32);
                        const uint64_t db =
                            sdesc_sw128(aS + part * L::S_PLANE + (ks >> 2) * L::S_ATOM + (ks & 3) * 32);
                        mma_bf16_ss(tmem + XC, da, db, idesc_bf16(128, 128), (part | ks) != 0);
                    }
                mma_commit(&bars[1]);
            }
        }
        __syncwarp();
        if (*sFlag == 0) warp0_wait(&bars[1], mma_phase, sFlag);
    }
    mma_phase ^= 1;
    __syncthreads();
    if (*sFlag) goto fail;
    tc_fence_after();
    // V (64 nodes x 128 columns bf16) by TMA into the space the products freed
    if (tid == 0) {
        v_issued = true;
        mbar_expect_tx(&bars[2], 2 * L::V_TILE);
        tma_load_4d(sm + L::VT, &tmV, &bars[2], 0, h, 0, b);
        tma_load_4d(sm + L::VT + L::V_TILE, &tmV, &bars[2], 64, h, 0, b);
    }

    // C rows (Q lanes) and G rows (K lanes) into shared memory: raw products,
    // then the decay (and beta) on the path entries, the only ones read
    // later; each warp takes 32 of the 64 columns.  W starts as the identity,
    // M as zero.
    {
        const bool qrow = row < 64;
        const int i = qrow ? row : row - 64;
        const int j0 = 32 * half;
        float* trow = (qrow ? sC : sG) + i * RS;
        uint32_t r[32];
        tmem_ld16(lane_base + AH + j0, *reinterpret_cast<uint32_t(*)[16]>(r));
        tmem_ld16(lane_base + AH + j0 + 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16));
        tmem_wait_ld();
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) trow[j0 + jj] = __uint_as_float(r[jj]);
        // decay (and beta for G) on this row's path entries in this half
        const float li = sL2[i];
        const float scale = qrow ? 1.f : sBeta[i];
        const uint64_t m = qrow ? sMask[i] : (sMask[i] & ~(1ull << i));
        for (uint32_t bits = uint32_t(m >> j0); bits; bits &= bits - 1) {
            const int j = j0 + __ffs(bits) - 1;
            trow[j] *= scale * exp2f(li - sL2[j]);
        }
        {
            for (int e = tid; e < TP * TP; e += NT) {
                const int a = e >> 6, c = e & 63;
                sW[a * RS + c] = (a == c) ? 1.f : 0.f;
                sM[a * RS + c] = 0.f;
            }
        }
    }
    __syncthreads();

    {
        // Finite Neumann series (Bole's solve) for W = sum_{m=0..d} (-G)^m on
        // tcgen05: P_0 = I, P_m = -G P_{m-1}, d rounds; G is the A operand in
        // tensor memory (K rows, tf32 hi + lo), P^T the B operand in shared
        // memory (tf32 hi + lo); each round is hi*hi + hi*lo + lo*hi.
        uint8_t* sPh = sm + L::PH;
        uint8_t* sPl = sm + L::PL;
        float wacc[32];  // K rows: this thread's 32 columns of its W row
        const int i = row - 64;
        const int jb = half * 32;
        if (quad >= 2) {
            // G row -> A hi/lo (K lanes, columns AH/AL); P_0 = I
            if (half == 0) {
                const uint64_t ms = sMask[i] & ~(1ull << i);
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t rh[16], rl[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = cb * 16 + jj;
                        const float x = ((ms >> j) & 1ull) ? sG[i * RS + j] : 0.f;
                        split_tf32(x, rh[jj], rl[jj]);
                    }
                    tmem_st16(lane_base + AH + cb * 16, rh);
                    tmem_st16(lane_base + AL + cb * 16, rl);
                }
                tmem_wait_st();
            }
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = jb + jj;
                const float x = (j == i) ? 1.f : 0.f;
                wacc[jj] = x;
                // P^T[n = j][k = i] (K-major, 64 rows)
                *reinterpret_cast<uint32_t*>(sPh + kmajor_tf32_off(j, i, 64)) = to_tf32(x);
                *reinterpret_cast<uint32_t*>(sPl + kmajor_tf32_off(j, i, 64)) = 0u;
            }
        }
        const int rounds = *sDmax;
        for (int m = 1; m <= rounds; ++m) {
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (warp == 0) {
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t aH = smem_u32(sPh), aL = smem_u32(sPl);
                    // G P into the spare columns
#pragma unroll
                    for (int pass = 0; pass < 3; ++pass)
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint32_t acol = (pass == 2 ? AL : AH) + ks * 8;
                            const uint32_t bb = (pass == 1 ? aL : aH) + (ks >> 2) * L::P_ATOM + (ks & 3) * 32;
                            mma_tf32_ts(tmem + YC, tmem + acol, sdesc_sw128(bb), idesc_tf32(128, 64),
                                        (pass | ks) != 0);
                        }
                    mma_commit(&bars[1]);
                }
                __syncwarp();
                warp0_wait(&bars[1], mma_phase, sFlag);
            }
            mma_phase ^= 1;
            __syncthreads();
            if (*sFlag) goto fail;
            tc_fence_after();
            if (quad >= 2) {
                uint32_t r[32];
                tmem_ld16(lane_base + YC + jb, *reinterpret_cast<uint32_t(*)[16]>(r));
                tmem_ld16(lane_base + YC + jb + 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16));
                tmem_wait_ld();
                const bool last = (m == rounds);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const float z = -__uint_as_float(r[jj]);
                    wacc[jj] += z;
                    if (!last) {
                        uint32_t zh, zl;
                        split_tf32(z, zh, zl);
                        *reinterpret_cast<uint32_t*>(sPh + kmajor_tf32_off(jb + jj, i, 64)) = zh;
                        *reinterpret_cast<uint32_t*>(sPl + kmajor_tf32_off(jb + jj, i, 64)) = zl;
                    }
                }
            }
        }
        if (quad >= 2) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) sW[i * RS + jb + jj] = wacc[jj];
        }
        __syncthreads();
        // M = C W: M_i. = sum_{k in path(i)} C_ik W_k. (zero off the paths,
        // since W_k. is); one warp per row, lanes over columns.
        for (int i2 = warp; i2 < TP; i2 += NT / 32) {
            const uint64_t pi = sMask[i2];
            const float* crow = sC + i2 * RS;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int wd = 0; wd < 2; ++wd) {
                uint32_t bits = uint32_t(pi >> (32 * wd));
                while (bits) {
                    const int k = 32 * wd + __ffs(bits) - 1;
                    bits &= bits - 1;
                    const float ck = crow[k];
                    a0 += ck * sW[k * RS + lane];
                    a1 += ck * sW[k * RS + lane + 32];
                }
            }
            sM[i2 * RS + lane] = a0;
            sM[i2 * RS + lane + 32] = a1;
        }
        __syncthreads();
    }


    {
        // [M; W] -> tensor memory as tf32 hi and lo; each warp takes 32 columns.
        {
            const bool qrow = row < 64;
            const int i = qrow ? row : row - 64;
            const float* trow = (qrow ? sM : sW) + i * RS;
            const uint64_t pm = sMask[i];
    #pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                const int j0 = 32 * half + 16 * cb;
                uint32_t rh[16], rl[16];
    #pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const float x = ((pm >> (j0 + jj)) & 1ull) ? trow[j0 + jj] : 0.f;
                    split_tf32(x, rh[jj], rl[jj]);
                }
                tmem_st16(lane_base + AH + j0, rh);
                tmem_st16(lane_base + AL + j0, rl);
            }
            tmem_wait_st();
        }
        __syncthreads();
    }

    // V must have landed (all threads check the same phase; bounded wait)
    if (!mbar_wait(&bars[2], 0)) *sFlag = 1;
    __syncthreads();
    if (*sFlag) goto fail;
    // Q lanes: gamma X_Q in place.  K lanes: R = beta (V - gamma X_K) -> R^T
    // hi/lo in shared memory, then zero X_K so the product below leaves U.
    {
        const bool qrow = row < 64;
        const int i = qrow ? row : row - 64;
        const float gi = sGam[i], bi = sBeta[i];
        uint8_t* sRh = sm + L::RH;
        uint8_t* sRl = sm + L::RL;
        // element (column c, node i) of the K-major R^T operand: atom i/32,
        // row c, 16-byte chunk ((i%32)/4) ^ (c%8), word i%4
        const int ibase = (i >> 5) * L::R_ATOM + ((i & 3) << 2);
        const int ichunk = (i & 31) >> 2;
        uint32_t vw[32];
        if (!qrow) {
            const uint8_t* vrow = sm + L::VT + half * L::V_TILE + i * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const uint4 x = *reinterpret_cast<const uint4*>(vrow + ((ch ^ (i & 7)) << 4));
                vw[4 * ch] = x.x;
                vw[4 * ch + 1] = x.y;
                vw[4 * ch + 2] = x.z;
                vw[4 * ch + 3] = x.w;
            }
        }
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
            const int c0 = 64 * half + cb * 16;
            uint32_t r[16];
            tmem_ld16(lane_base + XC + c0, r);
            tmem_wait_ld();
            if (qrow) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) r[jj] = __float_as_uint(gi * __uint_as_float(r[jj]));
            } else {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int cw = cb * 16 + jj;  // column within this warp's 64
                    const float vv = (cw & 1) ? bf16_hi(vw[cw >> 1]) : bf16_lo(vw[cw >> 1]);
                    const float rr = bi * (vv - gi * __uint_as_float(r[jj]));
                    uint32_t rh, rl;
                    split_tf32(rr, rh, rl);
                    const int c = c0 + jj;
                    const int off = ibase + c * 128 + ((ichunk ^ (c & 7)) << 4);
                    *reinterpret_cast<uint32_t*>(sRh + off) = rh;
                    *reinterpret_cast<uint32_t*>(sRl + off) = rl;
                    r[jj] = 0u;
                }
            }
            tmem_st16(lane_base + XC + c0, r);
        }
        tmem_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // X += [M; W] R with three tf32 products (hi*hi + hi*lo + lo*hi).
    if (warp == 0) {
        if (lane == 0) {
            tc_fence_after();
            const uint32_t aRh = smem_u32(sm + L::RH), aRl = smem_u32(sm + L::RL);
#pragma unroll
            for (int pass = 0; pass < 3; ++pass)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t acol = (pass == 2 ? AL : AH) + ks * 8;
                    const uint32_t bb = (pass == 1 ? aRl : aRh) + (ks >> 2) * L::R_ATOM + (ks & 3) * 32;
                    mma_tf32_ts(tmem + XC, tmem + acol, sdesc_sw128(bb), idesc_tf32(128, 128), 1);
                }
            mma_commit(&bars[1]);
        }
        __syncwarp();
        warp0_wait(&bars[1], mma_phase, sFlag);
    }
    mma_phase ^= 1;
    __syncthreads();
    if (*sFlag) goto fail;
    tc_fence_after();

    // Rows 0..63 are o, rows 64..127 are U.
    {
        const bool qrow = row < 64;
        const int i = qrow ? row : row - 64;
        const bool live = i < T;
        const size_t nb = ((size_t(b) * T + (live ? i : 0)) * H + h) * DV + 64 * half;
        const float sc = qrow ? p.scale : 1.f;  // o carries the scale on q, U does not
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
            uint32_t r[16];
            tmem_ld16(lane_base + XC + 64 * half + cb * 16, r);
            tmem_wait_ld();
            if (!live) continue;
            if (qrow && p.o_bf16) {
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const __nv_bfloat162 pr =
                        __floats2bfloat162_rn(sc * __uint_as_float(r[2 * e]), sc * __uint_as_float(r[2 * e + 1]));
                    w[e] = *reinterpret_cast<const uint32_t*>(&pr);
                }
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + nb + cb * 16);
                dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
                float* base = qrow ? static_cast<float*>(p.o) : p.U;
                float4* dst = reinterpret_cast<float4*>(base + nb + cb * 16);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_float4(sc * __uint_as_float(r[4 * e]), sc * __uint_as_float(r[4 * e + 1]),
                                         sc * __uint_as_float(r[4 * e + 2]), sc * __uint_as_float(r[4 * e + 3]));
            }
        }
    }
    goto teardown;

fail:
    if (tid == 0) {
        raise_err(p.err, CANOPY_DEVERR_TIMEOUT);
        mbar_wait(&bars[0], 0);  // let copies in flight land before leaving
        if (v_issued) mbar_wait(&bars[2], 0);
    }

teardown:
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemColsNeu);
}

}  // namespace tc

// ---------------------------------------------------------------------------
// Host side.

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// [B][T][H][128] bf16 (q, k or v) -> boxes of 64 (last dim) x 64 (nodes) with
// the 128-byte swizzle; nodes past T read as zero.
bool make_bf16_row_map(CUtensorMap* m, const void* base, int B, int T, int H) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {128, cuuint64_t(H), cuuint64_t(T), cuuint64_t(B)};
    const cuuint64_t strides[3] = {128 * 2, cuuint64_t(H) * 128 * 2, cuuint64_t(T) * H * 128 * 2};
    const cuuint32_t box[4] = {64, 1, 64, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Node rows of o or U ([B][T][H][128], fp32 or bf16) for tiled bulk stores:
// boxes of 32 node rows x 128 columns of one (stream, head), no swizzle
// (a [32][128] row-major staging tile).
bool make_row_store_map(CUtensorMap* m, void* base, int bf16, int B, int T, int H) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t es = bf16 ? 2 : 4;
    const cuuint64_t dims[4] = {128, cuuint64_t(H), cuuint64_t(T), cuuint64_t(B)};
    const cuuint64_t strides[3] = {128 * es, cuuint64_t(H) * 128 * es, cuuint64_t(T) * H * 128 * es};
    const cuuint32_t box[4] = {128, 1, 32, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// S0 [B][H][128][128] fp32 -> boxes of 32 columns x 128 rows with the
// 128-byte swizzle (one (stream, head) state is four boxes).
bool make_state_map(CUtensorMap* m, const float* base, int B, int H) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {128, 128, cuuint64_t(H), cuuint64_t(B)};
    const cuuint64_t strides[3] = {128 * 4, 128 * 128 * 4, cuuint64_t(H) * 128 * 128 * 4};
    const cuuint32_t box[4] = {32, 128, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static cudaError_t launch_neumann(const void* q, const void* k, const tc::Params& prm, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    if (!make_bf16_row_map(&mq, q, prm.B, prm.T, prm.HK) || !make_bf16_row_map(&mk, k, prm.B, prm.T, prm.HK) ||
        !make_bf16_row_map(&mv, prm.v, prm.B, prm.T, prm.H))
        return cudaErrorInvalidValue;
    const int smem = tc::Smem::TOTAL_NEU + 1024;
    static bool attr = false;
    if (!attr) {
        cudaError_t e =
            cudaFuncSetAttribute(tc::verify_neumann_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 grid(prm.H, prm.B);
    tc::verify_neumann_kernel<<<grid, tc::NT, smem, st>>>(mq, mk, mv, prm);
    return cudaGetLastError();
}

cudaError_t launch_verify_neumann(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                  const float* S0, const int32_t* parent, int T, int B, int H, int HK, void* o,
                                  int o_bf16, float scale, const Ws& ws, cudaStream_t st) {
    tc::Params prm;
    prm.v = static_cast<const __nv_bfloat16*>(v);
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
    prm.HK = HK;
    prm.scale = scale;
    return launch_neumann(q, k, prm, st);
}

}  // namespace canopy
