// Closed-form tree verify in fp32 on CUDA cores (the fp32 path, and every
// size the tensor-core kernel does not take).
//
// canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed form".
// Three launches after tree prep:
//   gram:  per (b, h, 16-node block) X_Q = S0 q_i and X_K = S0 k_i for the
//          block's rows, then gamma_i X_Q,i and R_i = beta_i (v_i -
//          gamma_i X_K,i) into scratch; and for every j on path(i):
//          G_ij = beta_i exp(l_i - l_j) k_i.k_j (j != i), C_ij = exp(l_i - l_j)
//          q_i.k_j into scratch [B][H][T][T] (other entries are never read);
//   solve: per (b, h), level by level (nodes of equal depth together):
//          u_i = R_i - sum_{j in A(i)} G_ij u_j (forward substitution over the
//          ancestor bitmask), o_i = gamma_i X_Q,i + sum_{j in path(i)} C_ij u_j.
// All arithmetic is fp32.
#include <algorithm>

#include "common.cuh"

namespace canopy {

namespace simt {

constexpr int ROWS = 16;

// Eight consecutive elements (16 or 32 bytes, aligned) as fp32.
__device__ inline void load8(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(v[e] << 16);
        x[2 * e + 1] = __uint_as_float(v[e] & 0xFFFF0000u);
    }
}
__device__ inline void load8(const float* p, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p), c = *reinterpret_cast<const float4*>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
}

template <typename InT, int DK, int DV>
__global__ void __launch_bounds__(256) gram_kernel(const InT* __restrict__ q, const InT* __restrict__ k,
                                                   const InT* __restrict__ v, const float* __restrict__ beta,
                                                   const float* __restrict__ S0, int T, int H, int HK, Ws ws) {
    constexpr int GROUPS = 256 / DV;          // row groups for the S0 products
    constexpr int RPG = ROWS / GROUPS;        // rows per group
    __shared__ float sq[ROWS][DK];
    __shared__ float sk[ROWS][DK];
    __shared__ float sS0[DV][33];
    __shared__ int sPathList[8][kMaxT];
    const int i0 = blockIdx.x * ROWS, h = blockIdx.y, b = blockIdx.z;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const size_t rowstride = size_t(HK) * DK;   // q and k rows: key heads
    const int hk = h / (H / HK);                // the key head this value head reads

    for (int e = t; e < ROWS * DK; e += 256) {
        const int r = e / DK, d = e % DK, i = i0 + r;
        float xq = 0.f, xk = 0.f;
        if (i < T) {
            const size_t off = (size_t(b) * T + i) * rowstride + size_t(hk) * DK + d;
            xq = to_f(q[off]);
            xk = to_f(k[off]);
        }
        sq[r][d] = xq;
        sk[r][d] = xk;
    }

    const int vcol = t % DV, grp = t / DV;
    float aq[RPG], ak[RPG];
#pragma unroll
    for (int r = 0; r < RPG; ++r) aq[r] = ak[r] = 0.f;
    const float* S0bh = S0 + (size_t(b) * H + h) * DV * DK;
    for (int dc = 0; dc < DK; dc += 32) {
        __syncthreads();
        for (int e = t; e < DV * 32; e += 256) {
            const int vv = e / 32, d = e % 32;
            sS0[vv][d] = S0bh[size_t(vv) * DK + dc + d];
        }
        __syncthreads();
#pragma unroll 4
        for (int d = 0; d < 32; ++d) {
            const float s = sS0[vcol][d];
#pragma unroll
            for (int r = 0; r < RPG; ++r) {
                aq[r] += s * sq[grp * RPG + r][dc + d];
                ak[r] += s * sk[grp * RPG + r][dc + d];
            }
        }
    }
#pragma unroll
    for (int r = 0; r < RPG; ++r) {
        const int i = i0 + grp * RPG + r;
        if (i < T) {
            const size_t n = (size_t(b) * T + i) * H + h;
            const float gam = expf(ws.l[n]);
            const float be = beta[n];
            const float vv = to_f(v[n * DV + vcol]);
            ws.xq[n * DV + vcol] = gam * aq[r];
            ws.rr[n * DV + vcol] = be * (vv - gam * ak[r]);
        }
    }

    // G and C along each root path: one warp per row; the row's path is
    // turned into a list, and each lane takes whole entries (a full dk-long
    // dot product per lane, so the entries of a deep path run in parallel).
    __syncthreads();
    int* plist = sPathList[warp];
    for (int r = warp; r < ROWS; r += 8) {
        const int i = i0 + r;
        if (i >= T) break;
        const size_t ni = (size_t(b) * T + i) * H + h;
        const float li = ws.l[ni], bi = beta[ni];
        const uint32_t* mrow = ws.mask + (size_t(b) * T + i) * ws.W;
        uint32_t word = (lane < ws.W) ? mrow[lane] : 0u;
        if (lane == (i >> 5)) word |= 1u << (i & 31);  // path(i) = A(i) + {i}
        const int cntw = __popc(word);
        int off = cntw;
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, off, sh);
            if (lane >= sh) off += y;
        }
        const int n = __shfl_sync(0xffffffffu, off, 31);
        off -= cntw;
        for (uint32_t bits = word; bits; bits &= bits - 1) plist[off++] = 32 * lane + __ffs(bits) - 1;
        __syncwarp();
        float* Grow = ws.gs + ((size_t(b) * H + h) * T + i) * T;
        float* Crow = ws.cs + ((size_t(b) * H + h) * T + i) * T;
        for (int p = lane; p < n; p += 32) {
            const int j = plist[p];
            const InT* kj = k + (size_t(b) * T + j) * rowstride + size_t(hk) * DK;
            float kk0 = 0.f, kk1 = 0.f, qk0 = 0.f, qk1 = 0.f;
#pragma unroll 2
            for (int d = 0; d < DK; d += 8) {
                float x[8];
                load8(kj + d, x);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    kk0 += sk[r][d + e] * x[e];
                    kk1 += sk[r][d + e + 1] * x[e + 1];
                    qk0 += sq[r][d + e] * x[e];
                    qk1 += sq[r][d + e + 1] * x[e + 1];
                }
            }
            const float gam = expf(li - ws.l[(size_t(b) * T + j) * H + h]);
            Grow[j] = (j == i) ? 0.f : bi * gam * (kk0 + kk1);
            Crow[j] = gam * (qk0 + qk1);
        }
        __syncwarp();
    }
}

constexpr int SOLVE_NT = 512;  // threads of the solve kernel
constexpr int CHN = 16;        // nodes staged at a time (in level order)
constexpr int PSTRIDE = 256;   // staged path entries per node (kMaxT)

// Shared-memory bytes of solve_level_kernel for T nodes and DV value columns.
__host__ __device__ constexpr size_t solve_smem(int T, int DV) {
    return size_t(T) * DV * 4 + size_t(3 * kMaxT + 1) * 4 + size_t(CHN) * 8 + size_t(CHN) * PSTRIDE * 12 + 16 +
           size_t(CHN) * DV * 8;
}

// Forward substitution level by level: all nodes of one depth depend only on
// shallower nodes, so they are solved together.  Per node i (in a level):
//   u_i = R_i - sum_{j in A(i)} G_ij u_j,
//   o_i = gamma_i X_Q,i + sum_{j in path(i)} C_ij u_j.
// One CTA per (stream, head): SOLVE_NT / DV groups of DV threads (one per
// value column); U of every solved node stays in shared memory.  Per chunk
// of CHN nodes in level order, one warp per node turns its ancestor bitmask
// into a list and stages (j, G_ij, C_ij); then the chunk's nodes are solved
// level by level, each group taking nodes of the level.
template <typename OutT, int DV>
__device__ __forceinline__ void level_solve(OutT* __restrict__ o, int T, int H, const Ws& ws, float scale) {
    constexpr int NG = SOLVE_NT / DV;
    extern __shared__ float smem[];
    float* sU = smem;                                       // [T][DV]
    int* sOrder = reinterpret_cast<int*>(sU + size_t(T) * DV);  // [kMaxT] nodes by depth
    int* sOff = sOrder + kMaxT;                             // [kMaxT + 1] level offsets
    int* sCnt = sOff + kMaxT + 1;                           // [kMaxT] nodes per level, then fill counters
    int* sNode = sCnt + kMaxT;                              // [CHN]
    int* sLen = sNode + CHN;                                // [CHN] ancestors staged per node
    int* sJ = sLen + CHN;                                   // [CHN][PSTRIDE]
    float* sG = reinterpret_cast<float*>(sJ + CHN * PSTRIDE);   // [CHN][PSTRIDE]
    float* sC = sG + CHN * PSTRIDE;                         // [CHN][PSTRIDE]; entry PSTRIDE-1 unused
    // [CHN][DV] R rows of the chunk (16-byte aligned for vector stores)
    float* sRr = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(sC + CHN * PSTRIDE) + 15) & ~uintptr_t(15));
    float* sXq = sRr + CHN * DV;                            // [CHN][DV] gamma X_Q rows of the chunk
    __shared__ float sCii[CHN];
    __shared__ int sMaxD;
    __shared__ float2 sPart[SOLVE_NT];  // per-thread partial sums when groups share a node
    const int h = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
    const int lane = t & 31, warp = t >> 5;
    const size_t bh = size_t(b) * H + h;

    for (int d = t; d < kMaxT; d += SOLVE_NT) sCnt[d] = 0;
    if (t == 0) sMaxD = 0;
    __syncthreads();
    int myd = 0;
    if (t < T) {
        myd = ws.depth[size_t(b) * T + t];
        myd = min(max(myd, 0), kMaxT - 1);
        atomicAdd(&sCnt[myd], 1);
        atomicMax(&sMaxD, myd);
    }
    __syncthreads();
    const int maxd = sMaxD;
    if (t == 0) {
        int acc = 0;
        for (int d = 0; d <= maxd; ++d) {
            sOff[d] = acc;
            acc += sCnt[d];
            sCnt[d] = 0;
        }
        sOff[maxd + 1] = acc;
    }
    __syncthreads();
    if (t < T) sOrder[sOff[myd] + atomicAdd(&sCnt[myd], 1)] = t;
    __syncthreads();

    const int c = t % DV, grp = t / DV;
    const float* gsb = ws.gs + bh * T * T;
    const float* csb = ws.cs + bh * T * T;
    // Chunks of CHN nodes in level order, across level boundaries: a chunk's
    // ancestor lists and coefficients are staged in one round (they depend
    // on nothing solved yet), then its nodes are solved level by level.
    int lv = 0;
    for (int c0 = 0; c0 < T; c0 += CHN) {
        const int cn = min(CHN, T - c0);
        // stage the chunk's ancestor lists and coefficients (one warp per node)
        if (warp < cn) {
            const int e = warp, i = sOrder[c0 + e];
            const uint32_t word = (lane < ws.W) ? ws.mask[(size_t(b) * T + i) * ws.W + lane] : 0u;
            const int cntw = __popc(word);
            int off = cntw;
#pragma unroll
            for (int sh = 1; sh < 32; sh <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, off, sh);
                if (lane >= sh) off += y;
            }
            const int n = __shfl_sync(0xffffffffu, off, 31);
            off -= cntw;
            int* jrow = sJ + e * PSTRIDE;
            for (uint32_t bits = word; bits; bits &= bits - 1) jrow[off++] = 32 * lane + __ffs(bits) - 1;
            __syncwarp();
            const float* grow = gsb + size_t(i) * T;
            const float* crow = csb + size_t(i) * T;
            // all of a lane's loads in flight at once (paths up to 256 long)
            for (int p0 = lane; p0 < n; p0 += 32 * 8) {
                int jj[8];
                float gv[8], cv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) jj[u] = (p0 + 32 * u < n) ? jrow[p0 + 32 * u] : i;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    gv[u] = grow[jj[u]];
                    cv[u] = crow[jj[u]];
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (p0 + 32 * u < n) {
                        sG[e * PSTRIDE + p0 + 32 * u] = gv[u];
                        sC[e * PSTRIDE + p0 + 32 * u] = cv[u];
                    }
            }
            if (lane == 0) {
                sNode[e] = i;
                sLen[e] = n;
                sCii[e] = crow[i];
            }
            // the node's R and gamma X_Q rows
            const size_t ni = (size_t(b) * T + i) * H + h;
            for (int cc = lane * 4; cc < DV; cc += 128) {
                *reinterpret_cast<float4*>(sRr + e * DV + cc) = *reinterpret_cast<const float4*>(ws.rr + ni * DV + cc);
                *reinterpret_cast<float4*>(sXq + e * DV + cc) = *reinterpret_cast<const float4*>(ws.xq + ni * DV + cc);
            }
        }
        __syncthreads();
        // the chunk's levels in order: positions [s0, s1) of level lv
        for (int s0 = 0; s0 < cn;) {
            while (sOff[lv + 1] <= c0 + s0) ++lv;
            const int s1 = min(cn, sOff[lv + 1] - c0);
            const int sn = s1 - s0;
            // groups per node: several groups share a node when the level
            // segment has fewer nodes than groups (deep trees: few nodes per
            // level, long paths); their partial sums meet in shared memory
            int gpn = 1;
            while (gpn * 2 * sn <= NG) gpn *= 2;
            if (gpn > 1) {
                const int e = s0 + grp / gpn, sub = grp % gpn;
                float acc = 0.f, out = 0.f;
                if (e < s1) {
                    const int n = sLen[e];
                    const int* jrow = sJ + e * PSTRIDE;
                    const float* gr = sG + e * PSTRIDE;
                    const float* cr = sC + e * PSTRIDE;
                    float a4[4] = {0.f, 0.f, 0.f, 0.f}, o4[4] = {0.f, 0.f, 0.f, 0.f};
                    int p = sub;
                    for (; p + 3 * gpn < n; p += 4 * gpn) {
                        int jq[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) jq[q] = jrow[p + q * gpn];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float u0 = sU[jq[q] * DV + c];
                            a4[q] -= gr[p + q * gpn] * u0;
                            o4[q] += cr[p + q * gpn] * u0;
                        }
                    }
                    for (; p < n; p += gpn) {
                        const float u0 = sU[jrow[p] * DV + c];
                        a4[0] -= gr[p] * u0;
                        o4[0] += cr[p] * u0;
                    }
                    acc = (a4[0] + a4[1]) + (a4[2] + a4[3]);
                    out = (o4[0] + o4[1]) + (o4[2] + o4[3]);
                }
                sPart[t] = make_float2(acc, out);
                __syncthreads();
                if (e < s1 && sub == 0) {
                    for (int q = 1; q < gpn; ++q) {
                        const float2 pq = sPart[t + q * DV];
                        acc += pq.x;
                        out += pq.y;
                    }
                    const int i = sNode[e];
                    const size_t ni = (size_t(b) * T + i) * H + h;
                    acc += sRr[e * DV + c];
                    out += sXq[e * DV + c] + sCii[e] * acc;
                    sU[i * DV + c] = acc;
                    ws.U[ni * DV + c] = acc;
                    store_out(o + ni * DV + c, scale * out);
                }
            } else {
                for (int e = s0 + grp; e < s1; e += NG) {
                    const int i = sNode[e], n = sLen[e];
                    const size_t ni = (size_t(b) * T + i) * H + h;
                    const int* jrow = sJ + e * PSTRIDE;
                    const float* gr = sG + e * PSTRIDE;
                    const float* cr = sC + e * PSTRIDE;
                    float acc = sRr[e * DV + c], out = sXq[e * DV + c];
                    float acc2 = 0.f, out2 = 0.f;
                    int p = 0;
                    for (; p + 1 < n; p += 2) {
                        const float u0 = sU[jrow[p] * DV + c], u1 = sU[jrow[p + 1] * DV + c];
                        acc -= gr[p] * u0;
                        out += cr[p] * u0;
                        acc2 -= gr[p + 1] * u1;
                        out2 += cr[p + 1] * u1;
                    }
                    if (p < n) {
                        const float u0 = sU[jrow[p] * DV + c];
                        acc -= gr[p] * u0;
                        out += cr[p] * u0;
                    }
                    acc += acc2;
                    out += out2 + sCii[e] * acc;
                    sU[i * DV + c] = acc;
                    ws.U[ni * DV + c] = acc;
                    store_out(o + ni * DV + c, scale * out);
                }
            }
            __syncthreads();
            s0 = s1;
        }
    }
}

template <typename OutT, int DV>
__global__ void __launch_bounds__(SOLVE_NT) solve_level_kernel(OutT* __restrict__ o, int T, int H, Ws ws,
                                                               float scale) {
    level_solve<OutT, DV>(o, T, H, ws, scale);
}

// Blocked forward substitution over 64-node diagonal blocks (canopy page,
// "Design decisions": 64-node diagonal blocks, off-diagonal updates as block
// products), for the G and C the tensor-core Gram kernel leaves: every tile
// on or below the diagonal written in full, zero off the paths.  For row
// block r:
//   R'_r = R_r - sum_{s<r} G_rs U_s,   W_rr = (I + G_rr)^-1,   U_r = W_rr R'_r,
//   O_r  = gamma X_Q,r + sum_{s<=r} C_rs U_s.
// W_rr has the in-block ancestor pattern; its row i follows from W (I + G) =
// I along i's in-block path, w_ik = [i = k] - sum_{e in path(i), e > k}
// w_ie G_ek, so the rows are independent and the depth of a block, not of the
// tree, sets the sequential part.  One CTA (512 threads) per (stream, head):
// thread (rg, cg) owns value columns 4 cg .. 4 cg + 3 of the block's rows
// 4 rg .. 4 rg + 3; U of the solved blocks stays in shared memory.  Trees
// shallower than BLOCK_MIN_DEPTH take the level-by-level substitution
// instead (fewer levels than the blocks cost, and it skips the zeros).
constexpr int BLK_NT = 512;
constexpr int BN = 64;     // nodes per block
constexpr int GS = 68;     // row stride of the staged 64 x 64 tiles (16-byte rows)
constexpr int BLOCK_MIN_DEPTH = 32;

// U is kept for whole blocks (rows past T are zero).
__host__ __device__ constexpr size_t block_smem(int T, int DV) {
    return size_t((T + BN - 1) / BN * BN) * DV * 4 + size_t(3) * BN * GS * 4 + size_t(BN) * DV * 4 +
           size_t(BN) * BN;
}

// 4 x 4 register tile: acc[r][c] -= or += sum_k A[4 rg + r][k] B[k][4 cg + c]
// over k = 0..63, A in a [BN][GS] tile, B in rows of DV floats (b = &B[0][4 cg]).
template <int DV, bool SUB>
__device__ __forceinline__ void tile_mac(float (&acc)[4][4], const float* a, const float* b) {
#pragma unroll 2
    for (int k = 0; k < BN; k += 4) {
        float4 u[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) u[kk] = *reinterpret_cast<const float4*>(b + (k + kk) * DV);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float4 w = *reinterpret_cast<const float4*>(a + r * GS + k);
            const float x = (w.x * u[0].x + w.y * u[1].x) + (w.z * u[2].x + w.w * u[3].x);
            const float y = (w.x * u[0].y + w.y * u[1].y) + (w.z * u[2].y + w.w * u[3].y);
            const float z = (w.x * u[0].z + w.y * u[1].z) + (w.z * u[2].z + w.w * u[3].z);
            const float q = (w.x * u[0].w + w.y * u[1].w) + (w.z * u[2].w + w.w * u[3].w);
            if (SUB) {
                acc[r][0] -= x; acc[r][1] -= y; acc[r][2] -= z; acc[r][3] -= q;
            } else {
                acc[r][0] += x; acc[r][1] += y; acc[r][2] += z; acc[r][3] += q;
            }
        }
    }
}

template <typename OutT, int DV>
__global__ void __launch_bounds__(BLK_NT, 1) solve_block_kernel(OutT* __restrict__ o, int T, int H, Ws ws,
                                                                float scale) {
    static_assert(DV == 128 && BLK_NT == 512 && SOLVE_NT == BLK_NT,
                  "thread tile: 16 row groups x 32 column groups of 4 x 4");
    __shared__ int sDepth;
    if (threadIdx.x == 0) sDepth = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < T; i += BLK_NT) atomicMax(&sDepth, ws.depth[size_t(blockIdx.y) * T + i]);
    __syncthreads();
    if (sDepth < BLOCK_MIN_DEPTH) {
        level_solve<OutT, DV>(o, T, H, ws, scale);
        return;
    }
    extern __shared__ float smem[];
    const int nb = (T + BN - 1) / BN;
    float* sU = smem;                  // [nb * BN][DV]
    float* sG = sU + size_t(nb) * BN * DV;   // [BN][GS] G tile
    float* sC = sG + BN * GS;          // [BN][GS] C tile
    float* sW = sC + BN * GS;          // [BN][GS] W_rr
    float* sRp = sW + BN * GS;         // [BN][DV] R'_r
    uint8_t* sPl = reinterpret_cast<uint8_t*>(sRp + BN * DV);  // [BN][BN] in-block paths, root side first
    const int h = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
    const int cg = t & 31, rg = t >> 5;  // columns 4 cg .. 4 cg + 3, block rows 4 rg .. 4 rg + 3
    const size_t bh = size_t(b) * H + h;
    const float* gsb = ws.gs + bh * T * T;
    const float* csb = ws.cs + bh * T * T;

    for (int r = 0; r < nb; ++r) {
        const int n0 = BN * r;
        float accR[4][4], accO[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = n0 + 4 * rg + q;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
            if (i < T) {
                const size_t ni = (size_t(b) * T + i) * H + h;
                x = *reinterpret_cast<const float4*>(ws.rr + ni * DV + 4 * cg);
                y = *reinterpret_cast<const float4*>(ws.xq + ni * DV + 4 * cg);
            }
            accR[q][0] = x.x; accR[q][1] = x.y; accR[q][2] = x.z; accR[q][3] = x.w;
            accO[q][0] = y.x; accO[q][1] = y.y; accO[q][2] = y.z; accO[q][3] = y.w;
        }
        // tiles s = 0..r of block row r; the off-diagonal ones update R' and O
        for (int s = 0; s <= r; ++s) {
            __syncthreads();  // the tiles of the previous step are no longer read
            for (int e = t; e < BN * BN; e += BLK_NT) {
                const int rho = e / BN, j = e % BN, i = n0 + rho, jj = BN * s + j;
                const bool in = i < T && jj < T;
                sG[rho * GS + j] = in ? gsb[size_t(i) * T + jj] : 0.f;
                sC[rho * GS + j] = in ? csb[size_t(i) * T + jj] : 0.f;
            }
            if (s == r && t < BN) {
                // in-block path of node n0 + t (ancestors in block r, then the node)
                const int rho = t, i = n0 + rho;
                uint64_t bits = 0;
                if (i < T) {
                    const uint32_t* mrow = ws.mask + (size_t(b) * T + i) * ws.W;
                    const uint32_t w0 = mrow[2 * r], w1 = (2 * r + 1 < ws.W) ? mrow[2 * r + 1] : 0u;
                    bits = (uint64_t(w1) << 32 | w0) | (1ull << rho);
                }
                int d = 0;
                for (; bits; bits &= bits - 1) sPl[rho * BN + d++] = uint8_t(__ffsll(static_cast<long long>(bits)) - 1);
                for (int z = d; z < BN; ++z) sPl[rho * BN + z] = 0xFF;
            }
            __syncthreads();
            if (s == r) break;
            const float* us = sU + size_t(BN) * s * DV + 4 * cg;
            tile_mac<DV, true>(accR, sG + 4 * rg * GS, us);
            tile_mac<DV, false>(accO, sC + 4 * rg * GS, us);
        }
        // W_rr rows (one thread per row), left-looking along the in-block path
        if (t < BN) {
            const int rho = t;
            const uint8_t* pl = sPl + rho * BN;
            float* wr = sW + rho * GS;
            for (int k = 0; k < BN; ++k) wr[k] = 0.f;
            int n = 0;
            while (n < BN && pl[n] != 0xFF) ++n;
            for (int d = n - 1; d >= 0; --d) {
                const int k = pl[d];
                float a0 = (d == n - 1) ? 1.f : 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
                int e = d + 1;
                for (; e + 3 < n; e += 4) {
                    const int e0 = pl[e], e1 = pl[e + 1], e2 = pl[e + 2], e3 = pl[e + 3];
                    a0 -= wr[e0] * sG[e0 * GS + k];
                    a1 -= wr[e1] * sG[e1 * GS + k];
                    a2 -= wr[e2] * sG[e2 * GS + k];
                    a3 -= wr[e3] * sG[e3 * GS + k];
                }
                for (; e < n; ++e) {
                    const int e0 = pl[e];
                    a0 -= wr[e0] * sG[e0 * GS + k];
                }
                wr[k] = (a0 + a1) + (a2 + a3);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
            *reinterpret_cast<float4*>(sRp + (4 * rg + q) * DV + 4 * cg) =
                make_float4(accR[q][0], accR[q][1], accR[q][2], accR[q][3]);
        __syncthreads();
        // U_r = W_rr R'_r (rows past T: zero W rows, zero R')
        float uo[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) uo[q][0] = uo[q][1] = uo[q][2] = uo[q][3] = 0.f;
        tile_mac<DV, false>(uo, sW + 4 * rg * GS, sRp + 4 * cg);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = n0 + 4 * rg + q;
            const float4 u4 = make_float4(uo[q][0], uo[q][1], uo[q][2], uo[q][3]);
            *reinterpret_cast<float4*>(sU + size_t(i) * DV + 4 * cg) = u4;
            if (i < T) *reinterpret_cast<float4*>(ws.U + ((size_t(b) * T + i) * H + h) * DV + 4 * cg) = u4;
        }
        __syncthreads();
        // O_r += C_rr U_r
        tile_mac<DV, false>(accO, sC + 4 * rg * GS, sU + size_t(n0) * DV + 4 * cg);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = n0 + 4 * rg + q;
            if (i < T) {
                OutT* op = o + ((size_t(b) * T + i) * H + h) * DV + 4 * cg;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) store_out(op + cc, scale * accO[q][cc]);
            }
        }
    }
}

}  // namespace simt

template <typename InT, int DK, int DV>
static cudaError_t launch_simt_typed(const void* q, const void* k, const void* v, const float* beta,
                                     const float* S0, int T, int B, int H, int HK, void* o, int o_bf16, float scale,
                                     const Ws& ws, int gram_done, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    if (!gram_done) {
        dim3 g1((T + simt::ROWS - 1) / simt::ROWS, H, B);
        simt::gram_kernel<InT, DK, DV><<<g1, 256, 0, st>>>(static_cast<const InT*>(q), static_cast<const InT*>(k),
                                                          static_cast<const InT*>(v), beta, S0, T, H, HK, ws);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    dim3 g2(H, B);
    if (gram_done) {
        // full tiles from the tensor-core Gram (dk = dv = 128): blocked substitution
        if constexpr (DV != 128) {
            return cudaErrorInvalidValue;
        } else {
            // either substitution may run (the CTA picks by its tree's depth)
            const size_t smem = std::max(simt::block_smem(T, DV), simt::solve_smem(T, DV));
            const size_t smem_max = std::max(simt::block_smem(kMaxT, DV), simt::solve_smem(kMaxT, DV));
            if (o_bf16) {
                static bool attr = false;
                if (!attr) {
                    e = cudaFuncSetAttribute(simt::solve_block_kernel<__nv_bfloat16, DV>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_max));
                    if (e != cudaSuccess) return e;
                    attr = true;
                }
                simt::solve_block_kernel<__nv_bfloat16, DV><<<g2, simt::BLK_NT, smem, st>>>(
                    static_cast<__nv_bfloat16*>(o), T, H, ws, scale);
            } else {
                static bool attr = false;
                if (!attr) {
                    e = cudaFuncSetAttribute(simt::solve_block_kernel<float, DV>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_max));
                    if (e != cudaSuccess) return e;
                    attr = true;
                }
                simt::solve_block_kernel<float, DV><<<g2, simt::BLK_NT, smem, st>>>(static_cast<float*>(o), T, H, ws,
                                                                                    scale);
            }
            return cudaGetLastError();
        }
    }
    const size_t smem = simt::solve_smem(T, DV);
    const size_t smem_max = simt::solve_smem(kMaxT, DV);
    if (o_bf16) {
        static bool attr = false;
        if (!attr) {
            e = cudaFuncSetAttribute(simt::solve_level_kernel<__nv_bfloat16, DV>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_max));
            if (e != cudaSuccess) return e;
            attr = true;
        }
        simt::solve_level_kernel<__nv_bfloat16, DV><<<g2, simt::SOLVE_NT, smem, st>>>(
            static_cast<__nv_bfloat16*>(o), T, H, ws, scale);
    } else {
        static bool attr = false;
        if (!attr) {
            e = cudaFuncSetAttribute(simt::solve_level_kernel<float, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     int(smem_max));
            if (e != cudaSuccess) return e;
            attr = true;
        }
        simt::solve_level_kernel<float, DV><<<g2, simt::SOLVE_NT, smem, st>>>(static_cast<float*>(o), T, H, ws,
                                                                              scale);
    }
    return cudaGetLastError();
}

cudaError_t launch_verify_simt(const void* q, const void* k, const void* v, int in_bf16, const float* beta,
                               const float* S0, int T, int B, int H, int HK, int d, void* o, int o_bf16, float scale,
                               const Ws& ws, int gram_done, cudaStream_t st) {
    using bf = __nv_bfloat16;
#define CANOPY_SIMT(IT, D) \
    return launch_simt_typed<IT, D, D>(q, k, v, beta, S0, T, B, H, HK, o, o_bf16, scale, ws, gram_done, st)
    if (d == 128) {
        if (in_bf16) CANOPY_SIMT(bf, 128);
        CANOPY_SIMT(float, 128);
    }
    if (in_bf16) CANOPY_SIMT(bf, 32);
    CANOPY_SIMT(float, 32);
#undef CANOPY_SIMT
}

}  // namespace canopy
