// Commit kernel: rebuild only the accepted node's state.
//
// canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed form"
// (last line) and "What the commit kernel stores", in the (dv, dk)
// orientation:  S_new = gamma_a S0 + sum_{j in path(a)} exp(l_a - l_j) u_j k_j^T,
// all in fp32, from the U and l the verify call left in the workspace and
// that call's k and parent.  Memory bound: every element of S0 is read once
// (one bulk copy per tile) and S_new written once with 16-byte coalesced
// stores; the path's k rows and weighted u entries are staged in shared
// memory 32 nodes at a time.
#include "common.cuh"

namespace canopy {

namespace cm {

constexpr int NT = 128;    // threads per CTA
constexpr int ROWS = 32;   // value rows per CTA
constexpr int CH = 32;     // path nodes staged per pass

__device__ inline float4 k4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ inline float4 k4(const __nv_bfloat16* p) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xFFFF0000u));
}

// One CTA rebuilds ROWS value rows of one (stream, head) state.  Its S0 tile
// is fetched by one bulk copy into shared memory at the start.  path(a) is
// walked up the stream's parent array (an input, so with state_ready it is
// read, and the path's k rows staged, while the preceding verify finishes);
// after that kernel has completed, one round of loads brings l and the u
// entries of the path, weighted by exp(l_a - l_j), and the path's rank-one
// terms are accumulated into the tile, which is stored in place of (or
// beside) S0.
template <typename InT, int DK, int DV>
__global__ void __launch_bounds__(NT) commit_kernel(const int32_t* __restrict__ accepted,
                                                    const int32_t* __restrict__ parent, const float* S0,
                                                    float* S_new, const InT* __restrict__ k, int T, int H, int HK,
                                                    Ws ws, int state_ready) {
    constexpr int C4 = DK / 4;             // float4 per state row (threads per row)
    constexpr int F4 = ROWS * C4 / NT;     // float4 per thread = rows per thread
    constexpr int KV = 16 / sizeof(InT);   // k elements per 16-byte load
    constexpr uint32_t TILE = ROWS * DK * 4;
    static_assert(F4 >= 2 && F4 % 2 == 0 && (ROWS * C4) % NT == 0 && NT % C4 == 0, "tile shape");
    __shared__ __align__(128) float sS[ROWS * DK];
    __shared__ __align__(16) InT sK[CH][DK];
    __shared__ __align__(16) float sWU[CH][ROWS];
    __shared__ int sPar[kMaxT];        // the stream's parents
    __shared__ int sPath[kMaxT];       // path(a), a first
    __shared__ __align__(8) uint64_t sBar;
    __shared__ int sN, sBad;
    const int rt = blockIdx.x, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
    const int v0 = rt * ROWS;
    const int hk = h / (H / HK);  // the key head this value head reads
    // this thread: rows r0 .. r0 + F4 - 1 of the tile, float4 column c4
    const int c4 = t % C4, r0 = (t / C4) * F4;
    const size_t sbase = ((size_t(b) * H + h) * DV + v0) * DK;

    // Programmatic dependent launch: with state_ready, the S0 tile, the
    // accepted node, the parents and the path's k rows are read while the
    // preceding kernel finishes; the workspace and S_new only after it has
    // completed.
    if (!state_ready) pdl_wait();
    pdl_trigger();
    if (t == 0) {
        mbar_init(&sBar, 1);
        fence_mbar_init();
        mbar_expect_tx(&sBar, TILE);
        bulk_load(sS, S0 + sbase, TILE, &sBar);
    }
    if (t < 32) {
        for (int j = t; j < T; j += 32) sPar[j] = parent[size_t(b) * T + j];
        int a = accepted[b];
        __syncwarp();
        if (t == 0) {
            const int bad = (a < -1 || a >= T) ? 1 : 0;
            if (bad) a = -1;
            // path(a) from a up to the root, parents sanitised as the verify
            // sanitises them (node 0 is the root; a parent outside [0, j)
            // reads as 0), so the walk ends within a + 1 steps
            int n = 0;
            for (int j = a; j >= 0;) {
                sPath[n++] = j;
                const int pj = sPar[j];
                j = (j == 0) ? -1 : ((pj >= 0 && pj < j) ? pj : 0);
            }
            sN = n;
            sBad = bad;
        }
    }
    __syncthreads();
    const int n = sN;
    // k rows of the first chunk of the path (an input)
    {
        const int cn = min(CH, n);
        for (int e = t; e < cn * (DK / KV); e += NT) {
            const int r = e / (DK / KV), c = (e % (DK / KV)) * KV, j = sPath[r];
            *reinterpret_cast<uint4*>(&sK[r][c]) =
                *reinterpret_cast<const uint4*>(k + ((size_t(b) * T + j) * HK + hk) * DK + c);
        }
    }
    if (state_ready) pdl_wait();
    if (sBad && t == 0 && h == 0 && rt == 0) raise_err(ws.err, CANOPY_DEVERR_ACCEPTED);
    const float la = (n > 0) ? ws.l[(size_t(b) * T + sPath[0]) * H + h] : 0.f;

    float4 acc[F4];
    bool have_tile = false;
    for (int c0 = 0; c0 == 0 || c0 < n; c0 += CH) {
        const int cn = max(0, min(CH, n - c0));
        if (c0) {
            __syncthreads();
            for (int e = t; e < cn * (DK / KV); e += NT) {
                const int r = e / (DK / KV), c = (e % (DK / KV)) * KV, j = sPath[c0 + r];
                *reinterpret_cast<uint4*>(&sK[r][c]) =
                    *reinterpret_cast<const uint4*>(k + ((size_t(b) * T + j) * HK + hk) * DK + c);
            }
        }
        for (int e = t; e < cn * ROWS; e += NT) {
            const int r = e / ROWS, c = e % ROWS, j = sPath[c0 + r];
            const size_t nh = (size_t(b) * T + j) * H + h;
            sWU[r][c] = expf(la - ws.l[nh]) * ws.U[nh * DV + v0 + c];
        }
        if (!have_tile) {
            if (!mbar_wait(&sBar, 0) && t == 0) raise_err(ws.err, CANOPY_DEVERR_TIMEOUT);
            const float gamma_a = (n > 0) ? expf(la) : 1.f;
#pragma unroll
            for (int u = 0; u < F4; ++u) {
                const float4 s = *reinterpret_cast<const float4*>(&sS[((r0 + u) * C4 + c4) * 4]);
                acc[u] = make_float4(gamma_a * s.x, gamma_a * s.y, gamma_a * s.z, gamma_a * s.w);
            }
            have_tile = true;
        }
        __syncthreads();
        for (int r = 0; r < cn; ++r) {
            const float4 kk = k4(&sK[r][c4 * 4]);
            float wu[F4];
#pragma unroll
            for (int u2 = 0; u2 < F4; u2 += 2) {
                const float2 w2 = *reinterpret_cast<const float2*>(&sWU[r][r0 + u2]);
                wu[u2] = w2.x;
                wu[u2 + 1] = w2.y;
            }
#pragma unroll
            for (int u = 0; u < F4; ++u) {
                acc[u].x += wu[u] * kk.x;
                acc[u].y += wu[u] * kk.y;
                acc[u].z += wu[u] * kk.z;
                acc[u].w += wu[u] * kk.w;
            }
        }
    }
#pragma unroll
    for (int u = 0; u < F4; ++u)
        *reinterpret_cast<float4*>(S_new + sbase + size_t((r0 + u) * C4 + c4) * 4) = acc[u];
}

}  // namespace cm

template <typename InT, int D>
static cudaError_t launch_commit_typed(const int32_t* accepted, const int32_t* parent, const float* S0,
                                       float* S_new, const void* k, int T, int B, int H, int HK, const Ws& ws,
                                       int state_ready, cudaStream_t st) {
    dim3 grid(D / cm::ROWS, H, B);
    return launch_pdl(cm::commit_kernel<InT, D, D>, grid, dim3(cm::NT), 0, st, accepted, parent, S0, S_new,
                      static_cast<const InT*>(k), T, H, HK, ws, state_ready);
}

cudaError_t launch_commit(const int32_t* accepted, const int32_t* parent, const float* S0, float* S_new,
                          const void* k, int in_bf16, int T, int B, int H, int HK, int d, const Ws& ws,
                          int state_ready, cudaStream_t st) {
    using bf = __nv_bfloat16;
    const int sr = state_ready;
    if (d == 128) {
        if (in_bf16) return launch_commit_typed<bf, 128>(accepted, parent, S0, S_new, k, T, B, H, HK, ws, sr, st);
        return launch_commit_typed<float, 128>(accepted, parent, S0, S_new, k, T, B, H, HK, ws, sr, st);
    }
    if (in_bf16) return launch_commit_typed<bf, 32>(accepted, parent, S0, S_new, k, T, B, H, HK, ws, sr, st);
    return launch_commit_typed<float, 32>(accepted, parent, S0, S_new, k, T, B, H, HK, ws, sr, st);
}

}  // namespace canopy
