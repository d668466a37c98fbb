// Closed-form tree verify on tcgen05 tensor cores (bf16 q/k/v, fp32 S0,
// fp32 accumulation in tensor memory), one 64-node block (T <= 64).
//
// Method: canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed
// form" (Bole's Theorem 1).  One CTA owns (stream b, head h, value tile of BV
// columns of the d_v x d_k state) and, for all T nodes:
//   1. tree prep: parent -> path bitmask, depth, l_i = sum log alpha (log2
//      units inside), by pointer jumping (common.cuh); nodes grouped by depth;
//   2. X  = [Q;K] S0_tile^T on tcgen05 (M = 128 rows = Q rows then K rows,
//      N = BV, K = dk); S0 is split into bf16 hi + lo parts in shared memory
//      so the product keeps ~16 mantissa bits of the fp32 state;
//      AC = [Q;K] K^T on tcgen05 (N = 64): rows 0..63 give Q K^T, rows
//      64..127 give K K^T;
//   3. epilogue (one thread per TMEM lane): C_ij = 2^(l2_i - l2_j) q_i.k_j and
//      G_ij = beta_i 2^(l2_i - l2_j) k_i.k_j on the root-path entries only,
//      R_i = beta_i (v_i - gamma_i X_K,i), all into shared memory;
//   4. the triangular solve (I + G) U = R in fp32, either level by level over
//      the tree (forward substitution; one warp per node, lanes over value
//      columns, sums over the ancestor bits) or as the finite Neumann series
//      on tcgen05 (Bole's solve, d rounds of Z <- -G Z);
//   5. O = gamma X_Q + C U in fp32, one warp per node, lanes over columns,
//      summing over path(i).
// Decay ratios are only ever 2^(l2_i - l2_j) with j on i's root path, so they
// lie in (0, 1] and never overflow ("Hard constraints", log-space gates).
#include "common.cuh"

namespace canopy {

namespace tc {

constexpr int DK = 128;
constexpr int DV = 128;
constexpr int TP = 64;   // nodes per block
constexpr int RS = 65;   // padded row stride (floats) of the T x T tables

template <int BV>
struct Smem {
    // phase A (until the first MMAs complete)
    static constexpr int QK = 0;                    // [Q;K] bf16: 2 atoms x 128 rows x 128 B
    static constexpr int S_ATOM = BV * 128;         // one 64-column bf16 atom of the S0 tile
    static constexpr int S_PLANE = 2 * S_ATOM;      // hi or lo plane
    static constexpr int S = 32768;                 // S0 hi then lo
    static constexpr int A_END = S + 2 * S_PLANE;
    // phase B (reuses phase A's space)
    static constexpr int GS = 0;                    // G fp32 [64][RS]; later gamma X_Q fp32 [64][BV+1]
    static constexpr int CS = GS + TP * RS * 4;     // C fp32 [64][RS]
    static constexpr int RR = CS + TP * RS * 4;     // R fp32 [64][BV+1]
    static constexpr int UR = RR + TP * (BV + 1) * 4;  // U fp32 [64][BV]
    static constexpr int ZT = 33792;                // Neumann: Z^T tf32 operand [BV][64] (1024-aligned)
    static constexpr int B_END = UR + TP * BV * 4;
    // small arrays
    static constexpr int SMALL = ((A_END > B_END ? A_END : B_END) + 255) & ~255;
    static constexpr int PAR = SMALL;               // int[64]   jump pointer
    static constexpr int LEN = PAR + 256;           // int[64]   path length
    static constexpr int L2 = LEN + 256;            // float[64] cumulative log2 gate
    static constexpr int GAM = L2 + 256;            // float[64] gamma = 2^l2
    static constexpr int BETA = GAM + 256;          // float[64]
    static constexpr int MASK = BETA + 256;         // u64[64]   path(i) incl. i
    static constexpr int BAR = MASK + 512;          // u64[2]
    static constexpr int TMEMSLOT = BAR + 16;       // u32
    static constexpr int FLAG = TMEMSLOT + 4;       // int
    static constexpr int DMAX = FLAG + 4;           // int: tree depth
    static constexpr int CNT = DMAX + 8;            // int[64]: nodes per depth level
    static constexpr int START = CNT + 256;         // int[65]: first slot of each level in LVL
    static constexpr int LVL = START + 272;         // int[64]: nodes sorted by depth
    static constexpr int TOTAL = LVL + 256;
    static_assert(ZT + BV * 256 <= SMALL, "Z^T placement");
    static_assert(TP * (BV + 1) * 4 <= TP * RS * 4 || BV == 64, "gamma X_Q placement");
};

// TMEM columns: X [0, BV), AC [BV, BV + 64); the Neumann variant adds
// Y [BV + 64, 2 BV + 64) for the per-round products G Z.
template <int BV, bool NEU>
__host__ __device__ constexpr uint32_t tmem_cols() {
    return (NEU && BV == 64) ? 256u : 128u;
}

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
};

__device__ inline float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ inline float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One element (column c, node i) of a K-major tf32 B operand [BV][64] in the
// 128-byte swizzle layout: node i sits in atom i/32, 16-byte chunk (i%32)/4.
template <int BV>
__device__ inline void store_zt(uint8_t* base, int c, int i, float x) {
    const int atom = i >> 5, chunk = (i & 31) >> 2;
    *reinterpret_cast<uint32_t*>(base + atom * (BV * 128) + c * 128 + ((chunk ^ (c & 7)) << 4) + ((i & 3) << 2)) =
        to_tf32(x);
}

// Raw 64-column AC row of this thread's TMEM lane into a padded smem row.
__device__ inline void ac_row_to_smem(uint32_t lane_base, int acol, float* row) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint32_t r[32];
        tmem_ld16(lane_base + acol + 32 * half, *reinterpret_cast<uint32_t(*)[16]>(r));
        tmem_ld16(lane_base + acol + 32 * half + 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16));
        tmem_wait_ld();
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) row[32 * half + jj] = __uint_as_float(r[jj]);
    }
}

// Bounded wait on an mbarrier phase by warp 0 only; the result is shared
// through sFlag and agreed on at the barrier that follows.
__device__ inline void warp0_wait(uint64_t* bar, uint32_t parity, int warp, int* sFlag) {
    if (warp == 0) {
        const bool ok = mbar_wait(bar, parity);
        if (!ok && (threadIdx.x & 31) == 0) *sFlag = 1;
    }
}

template <int BV, bool NEU>
__global__ void __launch_bounds__(128, 4)
    verify_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK, Params p) {
    using L = Smem<BV>;
    constexpr int NCC = BV / 32;  // value columns per lane
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
    int* sCnt = reinterpret_cast<int*>(sm + L::CNT);
    int* sStart = reinterpret_cast<int*>(sm + L::START);
    int* sLvl = reinterpret_cast<int*>(sm + L::LVL);
    float* sG = reinterpret_cast<float*>(sm + L::GS);
    float* sC = reinterpret_cast<float*>(sm + L::CS);
    float* sR = reinterpret_cast<float*>(sm + L::RR);
    float* sU = reinterpret_cast<float*>(sm + L::UR);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int vt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int T = p.T, H = p.H;
    const int v0 = vt * BV;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
        *sFlag = 0;
        *sDmax = 0;
    }
    if (warp == 0) {
        tmem_alloc(sTmem, tmem_cols<BV, NEU>());
        tmem_relinquish();
        tc_fence_before();
    }

    // S0 value tile: BV rows x 128 fp32, contiguous; 16-byte coalesced loads.
    constexpr int NS = BV / 4;
    float4 s0r[NS];
    {
        const float4* src = reinterpret_cast<const float4*>(p.S0 + ((size_t(b) * H + h) * DV + v0) * DK);
#pragma unroll
        for (int u = 0; u < NS; ++u) s0r[u] = __ldg(src + u * 128 + tid);
    }
    // Parents and gates; padded nodes get no path, beta = 0 and gamma = 1.
    uint32_t vw[BV / 2];
    int bad = 0;
    if (tid < TP) {
        const int i = tid;
        sCnt[i] = 0;
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

    uint8_t* sQK = sm + L::QK;
    if (tid == 0) {
        mbar_expect_tx(&bars[0], 4 * 64 * 64 * 2);
        tma_load_4d(sQK + 0, &tmQ, &bars[0], 0, h, 0, b);
        tma_load_4d(sQK + 16384, &tmQ, &bars[0], 64, h, 0, b);
        tma_load_4d(sQK + 8192, &tmK, &bars[0], 0, h, 0, b);
        tma_load_4d(sQK + 24576, &tmK, &bars[0], 64, h, 0, b);
    }

    // Tree prep (threads 0..63 own nodes; the whole CTA takes the barriers).
    jump_paths<1>(TP, sPtr, sLen, sL2, sMask);
    int rank = 0;
    if (tid < TP) {
        const int i = tid;
        if (i >= T) sMask[i] = 0ull;  // padded nodes: empty path
        sGam[i] = exp2f(sL2[i]);
        if (i < T) {
            atomicMax(sDmax, sLen[i] - 1);
            rank = atomicAdd(&sCnt[sLen[i] - 1], 1);
            if (vt == 0) p.l[(size_t(b) * T + i) * H + h] = sL2[i] * 0.69314718055994531f;
            if (vt == 0 && h == 0) {
                p.depth[size_t(b) * T + i] = sLen[i] - 1;
                const uint64_t strict = sMask[i] & ~(1ull << i);
                for (int w = 0; w < p.W; ++w)
                    p.mask[(size_t(b) * T + i) * p.W + w] = uint32_t(strict >> (32 * w));
            }
        }
    }
    __syncthreads();
    // Nodes grouped by depth level (order within a level is irrelevant: the
    // nodes of one level never depend on each other).
    if (warp == 0) {
        // exclusive scan of the level counts by one warp (levels < 64)
        const int dmax = *sDmax;
        int c0 = (lane <= dmax) ? sCnt[lane] : 0;
        int c1 = (lane + 32 <= dmax) ? sCnt[lane + 32] : 0;
        int x0 = c0, x1 = c1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y0 = __shfl_up_sync(0xffffffffu, x0, off);
            const int y1 = __shfl_up_sync(0xffffffffu, x1, off);
            if (lane >= off) {
                x0 += y0;
                x1 += y1;
            }
        }
        const int tot0 = __shfl_sync(0xffffffffu, x0, 31);
        const int tot1 = __shfl_sync(0xffffffffu, x1, 31);  // every lane takes part in the shuffle
        sStart[lane] = x0 - c0;
        sStart[lane + 32] = tot0 + x1 - c1;
        if (lane == 0) sStart[64] = tot0 + tot1;
    }
    __syncthreads();
    if (tid < T) sLvl[sStart[sLen[tid] - 1] + rank] = tid;

    // S0 tile -> bf16 hi and lo planes, K-major with the 128-byte swizzle.
    {
        uint8_t* sS = sm + L::S;
#pragma unroll
        for (int u = 0; u < NS; ++u) {
            const int f = u * 128 + tid;
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
    // V rows for the K-row threads (lane 64 + i holds node i): BV bf16;
    // issued here so their latency overlaps the first MMAs.
    {
        const int i = tid - 64;
        if (tid >= 64 && i < T) {
            const uint4* src = reinterpret_cast<const uint4*>(p.v + ((size_t(b) * T + i) * H + h) * DV + v0);
#pragma unroll
            for (int u = 0; u < BV / 8; ++u) {
                uint4 x = __ldg(src + u);
                vw[4 * u] = x.x;
                vw[4 * u + 1] = x.y;
                vw[4 * u + 2] = x.z;
                vw[4 * u + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int u = 0; u < BV / 2; ++u) vw[u] = 0;
        }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // First MMAs: X = [Q;K] (S0hi + S0lo)^T and AC = [Q;K] K^T.
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
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t da = sdesc_sw128(aQK + (ks >> 2) * 16384 + (ks & 3) * 32);
                        const uint64_t db =
                            sdesc_sw128(aS + part * L::S_PLANE + (ks >> 2) * L::S_ATOM + (ks & 3) * 32);
                        mma_bf16_ss(tmem, da, db, idesc_bf16(128, BV), (part | ks) != 0);
                    }
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t da = sdesc_sw128(aQK + (ks >> 2) * 16384 + (ks & 3) * 32);
                    const uint64_t db = sdesc_sw128(aQK + (ks >> 2) * 16384 + 8192 + (ks & 3) * 32);
                    mma_bf16_ss(tmem + BV, da, db, idesc_bf16(128, 64), ks != 0);
                }
                mma_commit(&bars[1]);
            }
        }
        __syncwarp();
        if (*sFlag == 0) warp0_wait(&bars[1], 0, warp, sFlag);
    }
    __syncthreads();
    if (*sFlag) {
        if (tid == 0) {
            raise_err(p.err, CANOPY_DEVERR_TIMEOUT);
            mbar_wait(&bars[0], 0);  // let copies in flight land before leaving
        }
        goto teardown;
    }
    tc_fence_after();

    {
        const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
        if (warp < 2) {
            // Q rows: C row i (raw Q K^T, then the decay on the path entries,
            // the only ones the output reads).
            const int i = tid;
            const float li = sL2[i];
            float* crow = sC + i * RS;
            ac_row_to_smem(lane_base, BV, crow);
            for (uint64_t bits = sMask[i]; bits; bits &= bits - 1) {
                const int j = __ffsll(static_cast<long long>(bits)) - 1;
                crow[j] *= exp2f(li - sL2[j]);
            }
        } else {
            const int i = tid - 64;
            const float li = sL2[i], bi = sBeta[i], gi = sGam[i];
            const uint64_t ms = sMask[i] & ~(1ull << i);
            if constexpr (!NEU) {
                // K rows: G row i on the strict ancestors, and R row i.
                float* grow = sG + i * RS;
                ac_row_to_smem(lane_base, BV, grow);
                for (uint64_t bits = ms; bits; bits &= bits - 1) {
                    const int j = __ffsll(static_cast<long long>(bits)) - 1;
                    grow[j] *= bi * exp2f(li - sL2[j]);
                }
                float* rrow = sR + i * (BV + 1);
#pragma unroll
                for (int cb = 0; cb < BV / 16; ++cb) {
                    uint32_t r[16];
                    tmem_ld16(lane_base + cb * 16, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int c = cb * 16 + jj;
                        const float vv = (c & 1) ? bf16_hi(vw[c >> 1]) : bf16_lo(vw[c >> 1]);
                        rrow[c] = bi * (vv - gi * __uint_as_float(r[jj]));
                    }
                }
            }
        }
    }

    if constexpr (!NEU) {
        __syncthreads();
        // Level-synchronous forward substitution over the tree (canopy page,
        // "The tree closed form", level-synchronous solve): the nodes of one
        // depth level depend only on shallower nodes, so each level is one
        // parallel step.  A warp takes a node, its lanes the value columns;
        // u_i = R_i - sum_{j in A(i)} G_ij u_j runs over the ancestor bits.
        const int dmax = *sDmax;
        for (int lv = 0; lv <= dmax; ++lv) {
            const int s1 = sStart[lv + 1];
            for (int idx = sStart[lv] + warp; idx < s1; idx += 4) {
                const int i = sLvl[idx];
                const float* grow = sG + i * RS;
                float a0[NCC], a1[NCC];
#pragma unroll
                for (int q = 0; q < NCC; ++q) {
                    a0[q] = sR[i * (BV + 1) + lane + 32 * q];
                    a1[q] = 0.f;
                }
                uint64_t bits = sMask[i] & ~(1ull << i);
                while (bits) {
                    const int j0 = __ffsll(static_cast<long long>(bits)) - 1;
                    bits &= bits - 1;
                    const float g0 = grow[j0];
                    const float* u0 = sU + j0 * BV + lane;
                    if (bits) {
                        const int j1 = __ffsll(static_cast<long long>(bits)) - 1;
                        bits &= bits - 1;
                        const float g1 = grow[j1];
                        const float* u1 = sU + j1 * BV + lane;
#pragma unroll
                        for (int q = 0; q < NCC; ++q) {
                            a0[q] -= g0 * u0[32 * q];
                            a1[q] -= g1 * u1[32 * q];
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < NCC; ++q) a0[q] -= g0 * u0[32 * q];
                    }
                }
                float* ug = p.U + ((size_t(b) * T + i) * H + h) * DV + v0 + lane;
#pragma unroll
                for (int q = 0; q < NCC; ++q) {
                    const float u = a0[q] + a1[q];
                    sU[i * BV + lane + 32 * q] = u;
                    ug[32 * q] = u;
                }
            }
            __syncthreads();
        }
    } else {
        // Finite Neumann series (Bole's solve): U = sum_{m=0..d} (-G)^m R.
        // Each round is one tcgen05 tf32 MMA, A = [.; G] read from TMEM (the
        // K rows of the AC block, overwritten with G), B = Z^T from shared
        // memory; rows 64..127 of the product are G Z_{m-1}, so
        // Z_m = -G Z_{m-1}.  d rounds for a tree of depth d.
        const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
        uint8_t* sZt = sm + L::ZT;
        float acc[BV];  // K rows: U row
        const int i = tid - 64;
        if (warp >= 2) {
            const float li = sL2[i], bi = sBeta[i], gi = sGam[i];
            const uint64_t ms = sMask[i] & ~(1ull << i);
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t r[16];
                tmem_ld16(lane_base + BV + cb * 16, r);
                tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int j = cb * 16 + jj;
                    const float gv = ((ms >> j) & 1ull) ? bi * __uint_as_float(r[jj]) * exp2f(li - sL2[j]) : 0.f;
                    r[jj] = to_tf32(gv);
                }
                tmem_st16(lane_base + BV + cb * 16, r);
            }
#pragma unroll
            for (int cb = 0; cb < BV / 16; ++cb) {
                uint32_t r[16];
                tmem_ld16(lane_base + cb * 16, r);
                tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int c = cb * 16 + jj;
                    const float vv = (c & 1) ? bf16_hi(vw[c >> 1]) : bf16_lo(vw[c >> 1]);
                    acc[c] = bi * (vv - gi * __uint_as_float(r[jj]));
                    store_zt<BV>(sZt, c, i, acc[c]);
                }
            }
            tmem_wait_st();
        }
        const int rounds = *sDmax;
        uint32_t parity = 1;
        for (int m = 1; m <= rounds; ++m) {
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (warp == 0) {
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t aZ = smem_u32(sZt);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t db = sdesc_sw128(aZ + (ks >> 2) * (BV * 128) + (ks & 3) * 32);
                        mma_tf32_ts(tmem + BV + 64, tmem + BV + ks * 8, db, idesc_tf32(128, BV), ks != 0);
                    }
                    mma_commit(&bars[1]);
                }
                __syncwarp();
                warp0_wait(&bars[1], parity, warp, sFlag);
            }
            parity ^= 1;
            __syncthreads();
            if (*sFlag) {
                if (tid == 0) raise_err(p.err, CANOPY_DEVERR_TIMEOUT);
                goto teardown;
            }
            tc_fence_after();
            if (warp >= 2) {
                const bool last = (m == rounds);
#pragma unroll
                for (int cb = 0; cb < BV / 16; ++cb) {
                    uint32_t r[16];
                    tmem_ld16(lane_base + BV + 64 + cb * 16, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int c = cb * 16 + jj;
                        const float z = -__uint_as_float(r[jj]);
                        acc[c] += z;
                        if (!last) store_zt<BV>(sZt, c, i, z);
                    }
                }
            }
        }
        __syncthreads();  // the last round's Z^T reads are done before sU overwrites
        if (warp >= 2) {
#pragma unroll
            for (int c = 0; c < BV; ++c) sU[i * BV + c] = acc[c];
            if (i < T) {
                float4* dst = reinterpret_cast<float4*>(p.U + ((size_t(b) * T + i) * H + h) * DV + v0);
#pragma unroll
                for (int e = 0; e < BV / 4; ++e)
                    dst[e] = make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2], acc[4 * e + 3]);
            }
        }
        __syncthreads();
    }

    // gamma X_Q rows into shared memory (over G, no longer needed) so that
    // the output can run with lanes over columns.
    if (warp < 2) {
        const int i = tid;
        const uint32_t lane_base = tmem + (uint32_t(warp * 32) << 16);
        const float gi = sGam[i];
        float* xrow = sG + i * (BV + 1);
#pragma unroll
        for (int cb = 0; cb < BV / 16; ++cb) {
            uint32_t r[16];
            tmem_ld16(lane_base + cb * 16, r);
            tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) xrow[cb * 16 + jj] = gi * __uint_as_float(r[jj]);
        }
    }
    __syncthreads();

    // Output on CUDA cores in fp32, one warp per node, lanes over columns:
    // o_i = gamma_i X_Q,i + sum_{j in path(i)} C_ij u_j.
    for (int i = warp; i < T; i += 4) {
        const float* crow = sC + i * RS;
        float a0[NCC], a1[NCC];
#pragma unroll
        for (int q = 0; q < NCC; ++q) {
            a0[q] = sG[i * (BV + 1) + lane + 32 * q];
            a1[q] = 0.f;
        }
        uint64_t bits = sMask[i];
        while (bits) {
            const int j0 = __ffsll(static_cast<long long>(bits)) - 1;
            bits &= bits - 1;
            const float c0 = crow[j0];
            const float* u0 = sU + j0 * BV + lane;
            if (bits) {
                const int j1 = __ffsll(static_cast<long long>(bits)) - 1;
                bits &= bits - 1;
                const float c1 = crow[j1];
                const float* u1 = sU + j1 * BV + lane;
#pragma unroll
                for (int q = 0; q < NCC; ++q) {
                    a0[q] += c0 * u0[32 * q];
                    a1[q] += c1 * u1[32 * q];
                }
            } else {
#pragma unroll
                for (int q = 0; q < NCC; ++q) a0[q] += c0 * u0[32 * q];
            }
        }
        const size_t ob = ((size_t(b) * T + i) * H + h) * DV + v0 + lane;
#pragma unroll
        for (int q = 0; q < NCC; ++q) {
            const float x = a0[q] + a1[q];
            if (p.o_bf16)
                static_cast<__nv_bfloat16*>(p.o)[ob + 32 * q] = __float2bfloat16_rn(x);
            else
                static_cast<float*>(p.o)[ob + 32 * q] = x;
        }
    }

teardown:
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, tmem_cols<BV, NEU>());
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

// [B][T][H][128] bf16 -> boxes of 64 (dk) x 64 (nodes) with the 128-byte swizzle.
static bool make_qk_map(CUtensorMap* m, const void* base, int B, int T, int H) {
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

template <int BV, bool NEU>
static cudaError_t launch_tc(const void* q, const void* k, const tc::Params& prm, cudaStream_t st) {
    CUtensorMap mq, mk;
    if (!make_qk_map(&mq, q, prm.B, prm.T, prm.H) || !make_qk_map(&mk, k, prm.B, prm.T, prm.H))
        return cudaErrorInvalidValue;
    const int smem = tc::Smem<BV>::TOTAL + 1024;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(tc::verify_kernel<BV, NEU>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 grid(tc::DV / BV, prm.H, prm.B);
    tc::verify_kernel<BV, NEU><<<grid, 128, smem, st>>>(mq, mk, prm);
    return cudaGetLastError();
}

cudaError_t launch_verify_tc(const void* q, const void* k, const void* v, const float* g, const float* beta,
                             const float* S0, const int32_t* parent, int T, int B, int H, void* o, int o_bf16,
                             const Ws& ws, int bv, int neumann, cudaStream_t st) {
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
    if (neumann) return launch_tc<32, true>(q, k, prm, st);
    if (bv == 64) return launch_tc<64, false>(q, k, prm, st);
    return launch_tc<32, false>(q, k, prm, st);
}

}  // namespace canopy
