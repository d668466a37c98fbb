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
//   solve: per (b, h), one thread per value column, nodes in index order:
//          u_i = R_i - sum_{j in A(i)} G_ij u_j (forward substitution over the
//          ancestor bitmask), o_i = gamma_i X_Q,i + sum_{j in path(i)} C_ij u_j.
// All arithmetic is fp32.
#include "common.cuh"

namespace canopy {

namespace simt {

constexpr int ROWS = 16;

template <typename InT, int DK, int DV>
__global__ void __launch_bounds__(256) gram_kernel(const InT* __restrict__ q, const InT* __restrict__ k,
                                                   const InT* __restrict__ v, const float* __restrict__ beta,
                                                   const float* __restrict__ S0, int T, int H, Ws ws) {
    constexpr int GROUPS = 256 / DV;          // row groups for the S0 products
    constexpr int RPG = ROWS / GROUPS;        // rows per group
    constexpr int EL = DK / 32;               // dk elements per lane
    __shared__ float sq[ROWS][DK];
    __shared__ float sk[ROWS][DK];
    __shared__ float sS0[DV][33];
    const int i0 = blockIdx.x * ROWS, h = blockIdx.y, b = blockIdx.z;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const size_t rowstride = size_t(H) * DK;

    for (int e = t; e < ROWS * DK; e += 256) {
        const int r = e / DK, d = e % DK, i = i0 + r;
        float xq = 0.f, xk = 0.f;
        if (i < T) {
            const size_t off = (size_t(b) * T + i) * rowstride + size_t(h) * DK + d;
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

    // G and C along each root path: one warp per row, lanes split dk.
    for (int r = warp; r < ROWS; r += 8) {
        const int i = i0 + r;
        if (i >= T) break;
        const size_t ni = (size_t(b) * T + i) * H + h;
        const float li = ws.l[ni], bi = beta[ni];
        float ki[EL], qi[EL];
#pragma unroll
        for (int e = 0; e < EL; ++e) {
            ki[e] = sk[r][lane * EL + e];
            qi[e] = sq[r][lane * EL + e];
        }
        const uint32_t* mrow = ws.mask + (size_t(b) * T + i) * ws.W;
        float* Grow = ws.gs + ((size_t(b) * H + h) * T + i) * T;
        float* Crow = ws.cs + ((size_t(b) * H + h) * T + i) * T;
        for (int w = 0; w <= (i >> 5); ++w) {
            uint32_t bits = (w < ws.W) ? mrow[w] : 0u;
            if (w == (i >> 5)) bits |= 1u << (i & 31);  // path(i) = A(i) + {i}
            while (bits) {
                const int j = 32 * w + __ffs(bits) - 1;
                bits &= bits - 1;
                const InT* kj = k + (size_t(b) * T + j) * rowstride + size_t(h) * DK + lane * EL;
                float kk = 0.f, qk = 0.f;
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    const float x = to_f(kj[e]);
                    kk += ki[e] * x;
                    qk += qi[e] * x;
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    kk += __shfl_xor_sync(0xffffffffu, kk, off);
                    qk += __shfl_xor_sync(0xffffffffu, qk, off);
                }
                if (lane == 0) {
                    const float gam = expf(li - ws.l[(size_t(b) * T + j) * H + h]);
                    Grow[j] = (j == i) ? 0.f : bi * gam * kk;
                    Crow[j] = gam * qk;
                }
            }
        }
    }
}

template <typename OutT, int DV>
__global__ void __launch_bounds__(128) solve_kernel(OutT* __restrict__ o, int T, int H, Ws ws) {
    extern __shared__ float sU[];  // [T][DV]
    const int h = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
    if (c >= DV) return;
    for (int i = 0; i < T; ++i) {
        const size_t n = (size_t(b) * T + i) * H + h;
        float acc = ws.rr[n * DV + c];
        float out = ws.xq[n * DV + c];
        const uint32_t* mrow = ws.mask + (size_t(b) * T + i) * ws.W;
        const float* Grow = ws.gs + ((size_t(b) * H + h) * T + i) * T;
        const float* Crow = ws.cs + ((size_t(b) * H + h) * T + i) * T;
        for (int w = 0; w < ws.W; ++w) {
            uint32_t bits = mrow[w];
            while (bits) {
                const int j = 32 * w + __ffs(bits) - 1;
                bits &= bits - 1;
                const float uj = sU[j * DV + c];
                acc -= Grow[j] * uj;
                out += Crow[j] * uj;
            }
        }
        sU[i * DV + c] = acc;
        ws.U[n * DV + c] = acc;
        out += Crow[i] * acc;
        store_out(o + n * DV + c, out);
    }
}

}  // namespace simt

template <typename InT, int DK, int DV>
static cudaError_t launch_simt_typed(const void* q, const void* k, const void* v, const float* beta,
                                     const float* S0, int T, int B, int H, void* o, int o_bf16, const Ws& ws,
                                     cudaStream_t st) {
    dim3 g1((T + simt::ROWS - 1) / simt::ROWS, H, B);
    simt::gram_kernel<InT, DK, DV><<<g1, 256, 0, st>>>(static_cast<const InT*>(q), static_cast<const InT*>(k),
                                                      static_cast<const InT*>(v), beta, S0, T, H, ws);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int smem = T * DV * 4;
    dim3 g2(H, B);
    if (o_bf16) {
        static bool attr = false;
        if (!attr) {
            e = cudaFuncSetAttribute(simt::solve_kernel<__nv_bfloat16, DV>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxT * DV * 4);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        simt::solve_kernel<__nv_bfloat16, DV><<<g2, DV, smem, st>>>(static_cast<__nv_bfloat16*>(o), T, H, ws);
    } else {
        static bool attr = false;
        if (!attr) {
            e = cudaFuncSetAttribute(simt::solve_kernel<float, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxT * DV * 4);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        simt::solve_kernel<float, DV><<<g2, DV, smem, st>>>(static_cast<float*>(o), T, H, ws);
    }
    return cudaGetLastError();
}

cudaError_t launch_verify_simt(const void* q, const void* k, const void* v, int in_bf16, const float* beta,
                               const float* S0, int T, int B, int H, int d, void* o, int o_bf16, const Ws& ws,
                               cudaStream_t st) {
    if (d == 128) {
        if (in_bf16)
            return launch_simt_typed<__nv_bfloat16, 128, 128>(q, k, v, beta, S0, T, B, H, o, o_bf16, ws, st);
        return launch_simt_typed<float, 128, 128>(q, k, v, beta, S0, T, B, H, o, o_bf16, ws, st);
    }
    if (in_bf16) return launch_simt_typed<__nv_bfloat16, 32, 32>(q, k, v, beta, S0, T, B, H, o, o_bf16, ws, st);
    return launch_simt_typed<float, 32, 32>(q, k, v, beta, S0, T, B, H, o, o_bf16, ws, st);
}

}  // namespace canopy
