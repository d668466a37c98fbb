// Commit kernel: rebuild only the accepted node's state.
//
// canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed form"
// (last line) and "What the commit kernel stores", in the (dv, dk)
// orientation:  S_new = gamma_a S0 + sum_{j in path(a)} exp(l_a - l_j) u_j k_j^T,
// all in fp32, from the U, l and ancestor mask the verify call left in the
// workspace.  Memory bound: every element of S0 is read once and S_new
// written once, with 16-byte coalesced accesses; the path's k rows and u
// entries are staged in shared memory 32 nodes at a time.
#include "common.cuh"

namespace canopy {

namespace cm {

constexpr int ROWS = 16;   // value rows per CTA
constexpr int CHUNK = 32;  // path nodes staged per pass

template <typename InT, int DK, int DV>
__global__ void __launch_bounds__(128) commit_kernel(const int32_t* __restrict__ accepted,
                                                     const float* S0, float* S_new,
                                                     const InT* __restrict__ k, int T, int H, Ws ws) {
    constexpr int F4 = ROWS * DK / 4 / 128;  // float4 per thread
    __shared__ int sPath[kMaxT];
    __shared__ int sCount;
    __shared__ float sW[CHUNK];
    __shared__ __align__(16) float sK[CHUNK][DK];
    __shared__ float sUj[CHUNK][ROWS];
    const int rt = blockIdx.x, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
    const int v0 = rt * ROWS;

    int a = accepted[b];
    if (a < -1 || a >= T) {
        if (t == 0 && h == 0 && rt == 0) raise_err(ws.err, CANOPY_DEVERR_ACCEPTED);
        a = -1;
    }
    if (t == 0) {
        int m = 0;
        if (a >= 0) {
            const uint32_t* mrow = ws.mask + (size_t(b) * T + a) * ws.W;
            for (int w = 0; w < ws.W; ++w) {
                uint32_t bits = mrow[w];
                while (bits) {
                    sPath[m++] = 32 * w + __ffs(bits) - 1;
                    bits &= bits - 1;
                }
            }
            sPath[m++] = a;
        }
        sCount = m;
    }
    __syncthreads();
    const int m = sCount;
    const float la = (a >= 0) ? ws.l[(size_t(b) * T + a) * H + h] : 0.f;
    const float gamma_a = (a >= 0) ? expf(la) : 1.f;

    const size_t sbase = ((size_t(b) * H + h) * DV + v0) * DK;
    float4 acc[F4];
#pragma unroll
    for (int u = 0; u < F4; ++u) {
        const float4 s = *reinterpret_cast<const float4*>(S0 + sbase + size_t(u * 128 + t) * 4);
        acc[u] = make_float4(gamma_a * s.x, gamma_a * s.y, gamma_a * s.z, gamma_a * s.w);
    }
    for (int c0 = 0; c0 < m; c0 += CHUNK) {
        const int cn = min(CHUNK, m - c0);
        __syncthreads();
        for (int e = t; e < cn * DK; e += 128) {
            const int r = e / DK, d = e % DK, j = sPath[c0 + r];
            sK[r][d] = to_f(k[((size_t(b) * T + j) * H + h) * DK + d]);
        }
        for (int e = t; e < cn * ROWS; e += 128) {
            const int r = e / ROWS, c = e % ROWS, j = sPath[c0 + r];
            sUj[r][c] = ws.U[((size_t(b) * T + j) * H + h) * DV + v0 + c];
        }
        if (t < cn) sW[t] = expf(la - ws.l[(size_t(b) * T + sPath[c0 + t]) * H + h]);
        __syncthreads();
        for (int r = 0; r < cn; ++r) {
            const float w = sW[r];
#pragma unroll
            for (int u = 0; u < F4; ++u) {
                const int f = u * 128 + t, row = f / (DK / 4), c4 = f % (DK / 4);
                const float wu = w * sUj[r][row];
                const float4 kk = *reinterpret_cast<const float4*>(&sK[r][c4 * 4]);
                acc[u].x += wu * kk.x;
                acc[u].y += wu * kk.y;
                acc[u].z += wu * kk.z;
                acc[u].w += wu * kk.w;
            }
        }
    }
#pragma unroll
    for (int u = 0; u < F4; ++u) *reinterpret_cast<float4*>(S_new + sbase + size_t(u * 128 + t) * 4) = acc[u];
}

}  // namespace cm

template <typename InT, int D>
static cudaError_t launch_commit_typed(const int32_t* accepted, const float* S0, float* S_new, const void* k,
                                       int T, int B, int H, const Ws& ws, cudaStream_t st) {
    dim3 grid(D / cm::ROWS, H, B);
    cm::commit_kernel<InT, D, D><<<grid, 128, 0, st>>>(accepted, S0, S_new, static_cast<const InT*>(k), T, H, ws);
    return cudaGetLastError();
}

cudaError_t launch_commit(const int32_t* accepted, const float* S0, float* S_new, const void* k, int in_bf16,
                          int T, int B, int H, int d, const Ws& ws, cudaStream_t st) {
    if (d == 128) {
        if (in_bf16) return launch_commit_typed<__nv_bfloat16, 128>(accepted, S0, S_new, k, T, B, H, ws, st);
        return launch_commit_typed<float, 128>(accepted, S0, S_new, k, T, B, H, ws, st);
    }
    if (in_bf16) return launch_commit_typed<__nv_bfloat16, 32>(accepted, S0, S_new, k, T, B, H, ws, st);
    return launch_commit_typed<float, 32>(accepted, S0, S_new, k, T, B, H, ws, st);
}

}  // namespace canopy
