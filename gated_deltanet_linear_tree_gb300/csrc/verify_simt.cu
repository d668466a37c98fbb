// Closed-form tree verify in fp32 on CUDA cores: the fp32 path (and the
// dk = dv = 32 heads), which the tensor-core kernels do not take.
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
                                                   const float* __restrict__ S0, const int32_t* __restrict__ lengths,
                                                   int Ts, int H, int HK, Ws ws) {
    constexpr int GROUPS = 256 / DV;          // row groups for the S0 products
    constexpr int RPG = ROWS / GROUPS;        // rows per group
    __shared__ float sq[ROWS][DK];
    __shared__ float sk[ROWS][DK];
    __shared__ float sS0[DV][33];
    __shared__ int sPathList[8][kMaxT];
    const int i0 = blockIdx.x * ROWS, h = blockIdx.y, b = blockIdx.z;
    int lbad = 0;  // (reported by tree prep)
    const int T = stream_len(lengths, b, Ts, &lbad);  // this stream's nodes; Ts is the stride
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const size_t rowstride = size_t(HK) * DK;   // q and k rows: key heads
    const int hk = h / (H / HK);                // the key head this value head reads

    for (int e = t; e < ROWS * DK; e += 256) {
        const int r = e / DK, d = e % DK, i = i0 + r;
        float xq = 0.f, xk = 0.f;
        if (i < T) {
            const size_t off = (size_t(b) * Ts + i) * rowstride + size_t(hk) * DK + d;
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
            const size_t n = (size_t(b) * Ts + i) * H + h;
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
        const size_t ni = (size_t(b) * Ts + i) * H + h;
        const float li = ws.l[ni], bi = beta[ni];
        const uint32_t* mrow = ws.mask + (size_t(b) * Ts + i) * ws.W;
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
        float* Grow = ws.gs + ((size_t(b) * H + h) * Ts + i) * Ts;
        float* Crow = ws.cs + ((size_t(b) * H + h) * Ts + i) * Ts;
        for (int p = lane; p < n; p += 32) {
            const int j = plist[p];
            const InT* kj = k + (size_t(b) * Ts + j) * rowstride + size_t(hk) * DK;
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
            const float gam = expf(li - ws.l[(size_t(b) * Ts + j) * H + h]);
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
__device__ __forceinline__ void level_solve(OutT* __restrict__ o, const int32_t* __restrict__ lengths, int Ts, int H,
                                            const Ws& ws, float scale) {
    constexpr int NG = SOLVE_NT / DV;
    extern __shared__ float smem[];
    float* sU = smem;                                       // [T][DV]
    int* sOrder = reinterpret_cast<int*>(sU + size_t(Ts) * DV);  // [kMaxT] nodes by depth
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
    int lbad = 0;  // (reported by tree prep)
    const int T = stream_len(lengths, b, Ts, &lbad);  // this stream's nodes; Ts is the stride

    for (int d = t; d < kMaxT; d += SOLVE_NT) sCnt[d] = 0;
    if (t == 0) sMaxD = 0;
    __syncthreads();
    int myd = 0;
    if (t < T) {
        myd = ws.depth[size_t(b) * Ts + t];
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
    const float* gsb = ws.gs + bh * Ts * Ts;
    const float* csb = ws.cs + bh * Ts * Ts;
    // Chunks of CHN nodes in level order, across level boundaries: a chunk's
    // ancestor lists and coefficients are staged in one round (they depend
    // on nothing solved yet), then its nodes are solved level by level.
    int lv = 0;
    for (int c0 = 0; c0 < T; c0 += CHN) {
        const int cn = min(CHN, T - c0);
        // stage the chunk's ancestor lists and coefficients (one warp per node)
        if (warp < cn) {
            const int e = warp, i = sOrder[c0 + e];
            const uint32_t word = (lane < ws.W) ? ws.mask[(size_t(b) * Ts + i) * ws.W + lane] : 0u;
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
            const float* grow = gsb + size_t(i) * Ts;
            const float* crow = csb + size_t(i) * Ts;
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
            const size_t ni = (size_t(b) * Ts + i) * H + h;
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
                    const size_t ni = (size_t(b) * Ts + i) * H + h;
                    acc += sRr[e * DV + c];
                    out += sXq[e * DV + c] + sCii[e] * acc;
                    sU[i * DV + c] = acc;
                    ws.U[ni * DV + c] = acc;
                    store_out(o + ni * DV + c, scale * out);
                }
            } else {
                for (int e = s0 + grp; e < s1; e += NG) {
                    const int i = sNode[e], n = sLen[e];
                    const size_t ni = (size_t(b) * Ts + i) * H + h;
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
__global__ void __launch_bounds__(SOLVE_NT) solve_level_kernel(OutT* __restrict__ o,
                                                               const int32_t* __restrict__ lengths, int T, int H, Ws ws,
                                                               float scale) {
    level_solve<OutT, DV>(o, lengths, T, H, ws, scale);
}

}  // namespace simt

template <typename InT, int DK, int DV>
static cudaError_t launch_simt_typed(const void* q, const void* k, const void* v, const float* beta,
                                     const float* S0, const int32_t* lengths, int T, int B, int H, int HK, void* o,
                                     int o_bf16, float scale, const Ws& ws, cudaStream_t st) {
    dim3 g1((T + simt::ROWS - 1) / simt::ROWS, H, B);
    simt::gram_kernel<InT, DK, DV><<<g1, 256, 0, st>>>(static_cast<const InT*>(q), static_cast<const InT*>(k),
                                                      static_cast<const InT*>(v), beta, S0, lengths, T, H, HK,
                                                      ws);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 g2(H, B);
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
            static_cast<__nv_bfloat16*>(o), lengths, T, H, ws, scale);
    } else {
        static bool attr = false;
        if (!attr) {
            e = cudaFuncSetAttribute(simt::solve_level_kernel<float, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     int(smem_max));
            if (e != cudaSuccess) return e;
            attr = true;
        }
        simt::solve_level_kernel<float, DV><<<g2, simt::SOLVE_NT, smem, st>>>(static_cast<float*>(o), lengths, T, H,
                                                                              ws,
                                                                              scale);
    }
    return cudaGetLastError();
}

cudaError_t launch_verify_simt(const void* q, const void* k, const void* v, int in_bf16, const float* beta,
                               const float* S0, const int32_t* lengths, int T, int B, int H, int HK, int d, void* o,
                               int o_bf16, float scale, const Ws& ws, cudaStream_t st) {
    using bf = __nv_bfloat16;
#define CANOPY_SIMT(IT, D) \
    return launch_simt_typed<IT, D, D>(q, k, v, beta, S0, lengths, T, B, H, HK, o, o_bf16, scale, ws, st)
    if (d == 128) {
        if (in_bf16) CANOPY_SIMT(bf, 128);
        CANOPY_SIMT(float, 128);
    }
    if (in_bf16) CANOPY_SIMT(bf, 32);
    CANOPY_SIMT(float, 32);
#undef CANOPY_SIMT
}

}  // namespace canopy
