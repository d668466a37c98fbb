// Verify of tiny trees by replaying every node's root path from S0.
//
// canopy page (projects.dotslasha.me/p/canopy.md), "Design decisions" (the
// serial path below the crossover, the closed form above it) and "The gated
// delta rule": for node i with root path j_0 = 0, ..., j_d = i,
//     S <- S0;  for each j on the path: coef = beta_j (v_j - g_j S k_j),
//               S <- g_j S + coef k_j^T
//     o_i = S (scale q_i),   u_i = coef of the last step (i itself),
// which is the serial replay without its snapshots: every node restarts
// from S0, so nodes are independent and nothing is stored between them.
// u_i is the closed form's pseudo-value (S_i = g_i S_p + u_i k_i^T), so the
// commit reads U and l from the workspace as after any verify.  For trees
// of a few nodes the closed form's fixed chain of dependent stages costs
// more than these few rank-one steps.  One CTA per (stream, value head,
// 16 value rows), 8 lanes per row (dk / 8 entries each, 3-step shuffle
// reductions); nodes share the CTA's copy of S0's rows.
#include "common.cuh"

namespace canopy {

namespace pr {

constexpr int ROWS = 16;
constexpr int MAXT = 8;  // trees this kernel takes

template <typename InT, typename OutT, int DK, int DV>
__global__ void __launch_bounds__(128) path_replay_kernel(const InT* __restrict__ q, const InT* __restrict__ k,
                                                          const InT* __restrict__ v, const float* __restrict__ g,
                                                          const float* __restrict__ beta,
                                                          const float* __restrict__ S0,
                                                          const int32_t* __restrict__ parent,
                                                          const int32_t* __restrict__ lengths, OutT* __restrict__ o,
                                                          int Ts, int H, int ratio, float scale, Ws ws) {
    constexpr int C4 = DK / 32;  // float4 chunks per lane
    __shared__ int sPar[MAXT];
    __shared__ float sA[MAXT], sB[MAXT];
    const int rt = blockIdx.x, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
    const int row = t >> 3, gl = t & 7;  // state row within the tile, lane within the row group
    const int vr = rt * ROWS + row;
    const int hk = (ratio == 1) ? h : h / ratio;  // the key head this value head reads

    // Ts is the stride of every [B][T] array, T this stream's node count
    int bad = 0;
    const int T = stream_len(lengths, b, Ts, &bad);
    if (t < T) {
        const int i = t;
        int p = parent[size_t(b) * Ts + i];
        if (!((i == 0) ? (p == -1) : (p >= 0 && p < i))) {
            bad |= CANOPY_DEVERR_TREE;
            p = (i == 0) ? -1 : 0;
        }
        float a = g[(size_t(b) * Ts + i) * H + h], be = beta[(size_t(b) * Ts + i) * H + h];
        if (!gate_ok(a, be)) {
            bad |= CANOPY_DEVERR_GATE;
            a = 1.f;
            be = 0.f;
        }
        sPar[i] = p;
        sA[i] = a;
        sB[i] = be;
    }
    if (bad && rt == 0) raise_err(ws.err, bad);
    __syncthreads();
    // tree outputs for the commit: l (natural log), depth, strict-ancestor mask
    if (rt == 0 && t < T) {
        const int i = t;
        float l = 0.f;
        int d = 0;
        uint32_t m = 0;
        for (int j = i; j >= 0; j = sPar[j]) {
            l += logf(sA[j]);
            if (j != i) {
                m |= 1u << j;
                ++d;
            }
        }
        ws.l[(size_t(b) * Ts + i) * H + h] = l;
        if (h == 0) {
            ws.depth[size_t(b) * Ts + i] = d;
            ws.mask[(size_t(b) * Ts + i) * ws.W] = m;  // T <= 8: one word
        }
    }

    float4 s0[C4];
    const float* S0row = S0 + ((size_t(b) * H + h) * DV + vr) * DK;
#pragma unroll
    for (int c = 0; c < C4; ++c) s0[c] = *reinterpret_cast<const float4*>(S0row + (c * 8 + gl) * 4);
    for (int i = 0; i < T; ++i) {
        // the root path of i, root first
        int path[MAXT];
        int n = 0;
        for (int j = i; j >= 0; j = sPar[j]) path[n++] = j;
        float4 s[C4];
#pragma unroll
        for (int c = 0; c < C4; ++c) s[c] = s0[c];
        float coef = 0.f;
        for (int e = n - 1; e >= 0; --e) {
            const int j = path[e];
            const size_t krow = (size_t(b) * Ts + j) * (H / ratio) + hk;
            float4 kk[C4];
#pragma unroll
            for (int c = 0; c < C4; ++c) kk[c] = load4(k + krow * DK + (c * 8 + gl) * 4);
            float sk = 0.f;
#pragma unroll
            for (int c = 0; c < C4; ++c) sk += s[c].x * kk[c].x + s[c].y * kk[c].y + s[c].z * kk[c].z + s[c].w * kk[c].w;
            sk += __shfl_xor_sync(0xffffffffu, sk, 4);
            sk += __shfl_xor_sync(0xffffffffu, sk, 2);
            sk += __shfl_xor_sync(0xffffffffu, sk, 1);
            const float a = sA[j], be = sB[j];
            const float vv = to_f(v[((size_t(b) * Ts + j) * H + h) * DV + vr]);
            coef = be * (vv - a * sk);
#pragma unroll
            for (int c = 0; c < C4; ++c) {
                s[c].x = a * s[c].x + coef * kk[c].x;
                s[c].y = a * s[c].y + coef * kk[c].y;
                s[c].z = a * s[c].z + coef * kk[c].z;
                s[c].w = a * s[c].w + coef * kk[c].w;
            }
        }
        const size_t nrow = (size_t(b) * Ts + i) * H + h;
        const size_t qrow = (size_t(b) * Ts + i) * (H / ratio) + hk;
        float4 qq[C4];
#pragma unroll
        for (int c = 0; c < C4; ++c) qq[c] = load4(q + qrow * DK + (c * 8 + gl) * 4);
        float oo = 0.f;
#pragma unroll
        for (int c = 0; c < C4; ++c) oo += s[c].x * qq[c].x + s[c].y * qq[c].y + s[c].z * qq[c].z + s[c].w * qq[c].w;
        oo += __shfl_xor_sync(0xffffffffu, oo, 4);
        oo += __shfl_xor_sync(0xffffffffu, oo, 2);
        oo += __shfl_xor_sync(0xffffffffu, oo, 1);
        if (gl == 0) {
            store_out(o + nrow * DV + vr, scale * oo);
            ws.U[nrow * DV + vr] = coef;
        }
    }
}

}  // namespace pr

template <typename InT, typename OutT, int D>
static cudaError_t launch_pr_typed(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                   const float* S0, const int32_t* parent, const int32_t* lengths, int T, int B, int H,
                                   int HK, void* o, float scale, const Ws& ws, cudaStream_t st) {
    dim3 grid(D / pr::ROWS, H, B);
    pr::path_replay_kernel<InT, OutT, D, D><<<grid, 128, 0, st>>>(
        static_cast<const InT*>(q), static_cast<const InT*>(k), static_cast<const InT*>(v), g, beta, S0, parent,
        lengths, static_cast<OutT*>(o), T, H, H / HK, scale, ws);
    return cudaGetLastError();
}

int path_replay_max_t() { return pr::MAXT; }

cudaError_t launch_path_replay(const void* q, const void* k, const void* v, int in_bf16, const float* g,
                               const float* beta, const float* S0, const int32_t* parent, const int32_t* lengths,
                               int T, int B, int H, int HK, int d, void* o, int o_bf16, float scale, const Ws& ws,
                               cudaStream_t st) {
    if (T > pr::MAXT) return cudaErrorInvalidValue;
#define CANOPY_PR(IT, OT, D) \
    return launch_pr_typed<IT, OT, D>(q, k, v, g, beta, S0, parent, lengths, T, B, H, HK, o, scale, ws, st)
    using bf = __nv_bfloat16;
    if (d == 128) {
        if (in_bf16) {
            if (o_bf16) CANOPY_PR(bf, bf, 128);
            CANOPY_PR(bf, float, 128);
        }
        if (o_bf16) CANOPY_PR(float, bf, 128);
        CANOPY_PR(float, float, 128);
    }
    if (in_bf16) {
        if (o_bf16) CANOPY_PR(bf, bf, 32);
        CANOPY_PR(bf, float, 32);
    }
    if (o_bf16) CANOPY_PR(float, bf, 32);
    CANOPY_PR(float, float, 32);
#undef CANOPY_PR
}

}  // namespace canopy
