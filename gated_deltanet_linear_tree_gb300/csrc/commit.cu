// Commit kernel: rebuild only the accepted node's state.
//
// canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed form"
// (last line) and "What the commit kernel stores", in the (dv, dk)
// orientation:  S_new = gamma_a S0 + sum_{j in path(a)} exp(l_a - l_j) u_j k_j^T,
// all in fp32, from the U, l and ancestor mask the verify call left in the
// workspace.  Memory bound: every element of S0 is read once and S_new
// written once, with 16-byte coalesced accesses issued before anything that
// depends on the accepted node; the path's k rows and weighted u entries are
// staged in shared memory 32 nodes at a time.
#include "common.cuh"

namespace canopy {

namespace cm {

constexpr int NT = 128;    // threads per CTA
constexpr int ROWS = 32;   // value rows per CTA
constexpr int CH = 32;     // path nodes staged per pass

// 16 bytes of a k row -> fp32 in shared memory
__device__ inline void stage_k16(float* dst, const float* src) {
    *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(src);
}
__device__ inline void stage_k16(float* dst, const __nv_bfloat16* src) {
    const uint4 w = *reinterpret_cast<const uint4*>(src);
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        dst[2 * e] = __uint_as_float(x[e] << 16);
        dst[2 * e + 1] = __uint_as_float(x[e] & 0xFFFF0000u);
    }
}

// One CTA rebuilds ROWS value rows of one (stream, head) state.  The S0 tile
// is requested first; meanwhile warp 0 turns the accepted node's ancestor
// bitmask into a node list (one 32-bit word per lane, offsets by a warp
// prefix sum); then the path's k rows and exp(l_a - l_j) u_j entries are
// staged in shared memory and accumulated into the tile, which is stored in
// place of (or beside) S0.
template <typename InT, int DK, int DV>
__global__ void __launch_bounds__(NT, 8) commit_kernel(const int32_t* __restrict__ accepted, const float* S0,
                                                       float* S_new, const InT* __restrict__ k, int T, int H,
                                                       Ws ws) {
    constexpr int C4 = DK / 4;             // float4 per state row
    constexpr int F4 = ROWS * C4 / NT;     // float4 per thread
    constexpr int KV = 16 / sizeof(InT);   // k elements per 16-byte load
    static_assert(F4 >= 1 && (ROWS * C4) % NT == 0 && NT % C4 == 0, "tile shape");
    __shared__ int sPath[kMaxT];
    __shared__ int sN;
    __shared__ float sLa;
    __shared__ __align__(16) float sK[CH][DK];
    __shared__ float sWU[CH][ROWS];
    const int rt = blockIdx.x, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
    const int v0 = rt * ROWS;

    const size_t sbase = ((size_t(b) * H + h) * DV + v0) * DK;
    float4 acc[F4];
#pragma unroll
    for (int u = 0; u < F4; ++u) acc[u] = *reinterpret_cast<const float4*>(S0 + sbase + size_t(u * NT + t) * 4);

    if (t < 32) {
        int a = accepted[b];
        if (a < -1 || a >= T) {
            if (t == 0 && h == 0 && rt == 0) raise_err(ws.err, CANOPY_DEVERR_ACCEPTED);
            a = -1;
        }
        int n = 0;
        float la = 0.f;
        if (a >= 0) {
            const uint32_t word = (t < ws.W) ? ws.mask[(size_t(b) * T + a) * ws.W + t] : 0u;
            const int c = __popc(word);
            int off = c;
#pragma unroll
            for (int sh = 1; sh < 32; sh <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, off, sh);
                if (t >= sh) off += y;
            }
            n = __shfl_sync(0xffffffffu, off, 31) + 1;
            off -= c;
            for (uint32_t bits = word; bits; bits &= bits - 1) sPath[off++] = 32 * t + __ffs(bits) - 1;
            la = ws.l[(size_t(b) * T + a) * H + h];
            if (t == 0) sPath[n - 1] = a;
        }
        if (t == 0) {
            sN = n;
            sLa = la;
        }
    }
    __syncthreads();
    const int n = sN;
    const float la = sLa;
    const float gamma_a = (n > 0) ? expf(la) : 1.f;
#pragma unroll
    for (int u = 0; u < F4; ++u) {
        acc[u].x *= gamma_a;
        acc[u].y *= gamma_a;
        acc[u].z *= gamma_a;
        acc[u].w *= gamma_a;
    }

    for (int c0 = 0; c0 < n; c0 += CH) {
        const int cn = min(CH, n - c0);
        if (c0) __syncthreads();
        for (int e = t; e < cn * (DK / KV); e += NT) {
            const int r = e / (DK / KV), c = (e % (DK / KV)) * KV, j = sPath[c0 + r];
            stage_k16(&sK[r][c], k + ((size_t(b) * T + j) * H + h) * DK + c);
        }
        for (int e = t; e < cn * ROWS; e += NT) {
            const int r = e / ROWS, c = e % ROWS, j = sPath[c0 + r];
            const size_t nh = (size_t(b) * T + j) * H + h;
            sWU[r][c] = expf(la - ws.l[nh]) * ws.U[nh * DV + v0 + c];
        }
        __syncthreads();
        for (int r = 0; r < cn; ++r) {
#pragma unroll
            for (int u = 0; u < F4; ++u) {
                const int f = u * NT + t, row = f / C4, c4 = f % C4;
                const float wu = sWU[r][row];
                const float4 kk = *reinterpret_cast<const float4*>(&sK[r][c4 * 4]);
                acc[u].x += wu * kk.x;
                acc[u].y += wu * kk.y;
                acc[u].z += wu * kk.z;
                acc[u].w += wu * kk.w;
            }
        }
    }
#pragma unroll
    for (int u = 0; u < F4; ++u) *reinterpret_cast<float4*>(S_new + sbase + size_t(u * NT + t) * 4) = acc[u];
}

}  // namespace cm

template <typename InT, int D>
static cudaError_t launch_commit_typed(const int32_t* accepted, const float* S0, float* S_new, const void* k,
                                       int T, int B, int H, const Ws& ws, cudaStream_t st) {
    dim3 grid(D / cm::ROWS, H, B);
    cm::commit_kernel<InT, D, D><<<grid, cm::NT, 0, st>>>(accepted, S0, S_new, static_cast<const InT*>(k), T, H, ws);
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
