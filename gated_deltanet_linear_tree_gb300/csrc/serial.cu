// Serial parent-pointer replay: the crossover opponent.
//
// canopy page (projects.dotslasha.me/p/canopy.md), "Design decisions",
// serial baseline (SGLang's snapshot path): one program per (stream, head,
// value tile) walks the nodes in index order, takes its parent's state from
// a per-node snapshot buffer (or S0 for the root), applies one step of the
// gated delta rule in fp32,
//     S_i = alpha_i S_p (I - beta_i k_i k_i^T) + beta_i v_i k_i^T,  o_i = S_i (scale q_i),
// and writes the node's output.  Two choices keep it an honest opponent:
// the state of node i-1 stays in registers, so a node whose parent is i-1
// reads nothing back, and a snapshot is written only for nodes that have a
// child other than i+1.  A CTA holds 16 state rows, 8 lanes per row; each
// lane keeps dk/8 entries, so row dot products are 3-step shuffle reductions.
#include "common.cuh"

namespace canopy {

namespace serial {

constexpr int ROWS = 16;

template <typename InT, typename OutT, int DK, int DV>
__global__ void __launch_bounds__(128) replay_kernel(const InT* __restrict__ q, const InT* __restrict__ k,
                                                     const InT* __restrict__ v, const float* __restrict__ g,
                                                     const float* __restrict__ beta, const float* __restrict__ S0,
                                                     const int32_t* __restrict__ parent, OutT* __restrict__ o,
                                                     float* snap, int T, int H, int HK, float scale, int32_t* err) {
    constexpr int C4 = DK / 32;  // float4 chunks per lane
    __shared__ int sPar[kMaxT];
    __shared__ int sSnap[kMaxT];
    __shared__ float sA[kMaxT];
    __shared__ float sB[kMaxT];
    const int rt = blockIdx.x, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
    const int row = t >> 3, gl = t & 7;  // state row within the tile, lane within the row group
    const int vr = rt * ROWS + row;
    const int hk = h / (H / HK);  // the key head this value head reads

    int bad = 0;
    for (int i = t; i < T; i += blockDim.x) {
        int p = parent[size_t(b) * T + i];
        if (!((i == 0) ? (p == -1) : (p >= 0 && p < i))) {
            bad |= CANOPY_DEVERR_TREE;
            p = (i == 0) ? -1 : 0;
        }
        float a = g[(size_t(b) * T + i) * H + h], be = beta[(size_t(b) * T + i) * H + h];
        if (!gate_ok(a, be)) {
            bad |= CANOPY_DEVERR_GATE;
            a = 1.f;
            be = 0.f;
        }
        sPar[i] = p;
        sA[i] = a;
        sB[i] = be;
        sSnap[i] = 0;
    }
    if (bad && rt == 0) raise_err(err, bad);
    __syncthreads();
    for (int i = 1 + t; i < T; i += blockDim.x)
        if (sPar[i] != i - 1) sSnap[sPar[i]] = 1;  // a later node other than i+1 reads it
    __syncthreads();

    float4 s[C4];
    const float* S0row = S0 + ((size_t(b) * H + h) * DV + vr) * DK;
    for (int i = 0; i < T; ++i) {
        const int p = sPar[i];
        if (p < 0 || p != i - 1) {
            const float* src = (p < 0) ? S0row : snap + (((size_t(b) * T + p) * H + h) * DV + vr) * DK;
#pragma unroll
            for (int c = 0; c < C4; ++c) s[c] = *reinterpret_cast<const float4*>(src + (c * 8 + gl) * 4);
        }
        const size_t nrow = (size_t(b) * T + i) * H + h;
        const size_t krow = (size_t(b) * T + i) * HK + hk;
        float4 kk[C4], qq[C4];
#pragma unroll
        for (int c = 0; c < C4; ++c) {
            kk[c] = load4(k + krow * DK + (c * 8 + gl) * 4);
            qq[c] = load4(q + krow * DK + (c * 8 + gl) * 4);
        }
        const float a = sA[i], be = sB[i];
        const float vv = to_f(v[nrow * DV + vr]);
        float sk = 0.f;
#pragma unroll
        for (int c = 0; c < C4; ++c) sk += s[c].x * kk[c].x + s[c].y * kk[c].y + s[c].z * kk[c].z + s[c].w * kk[c].w;
        sk += __shfl_xor_sync(0xffffffffu, sk, 4);
        sk += __shfl_xor_sync(0xffffffffu, sk, 2);
        sk += __shfl_xor_sync(0xffffffffu, sk, 1);
        // S_i row = a * (s - be (s.k) k) + be v k
        const float coef = be * vv - a * be * sk;
        float oo = 0.f;
#pragma unroll
        for (int c = 0; c < C4; ++c) {
            s[c].x = a * s[c].x + coef * kk[c].x;
            s[c].y = a * s[c].y + coef * kk[c].y;
            s[c].z = a * s[c].z + coef * kk[c].z;
            s[c].w = a * s[c].w + coef * kk[c].w;
            oo += s[c].x * qq[c].x + s[c].y * qq[c].y + s[c].z * qq[c].z + s[c].w * qq[c].w;
        }
        oo += __shfl_xor_sync(0xffffffffu, oo, 4);
        oo += __shfl_xor_sync(0xffffffffu, oo, 2);
        oo += __shfl_xor_sync(0xffffffffu, oo, 1);
        if (gl == 0) store_out(o + nrow * DV + vr, scale * oo);
        if (sSnap[i]) {
            float* dst = snap + ((nrow)*DV + vr) * DK;
#pragma unroll
            for (int c = 0; c < C4; ++c) *reinterpret_cast<float4*>(dst + (c * 8 + gl) * 4) = s[c];
        }
    }
}

}  // namespace serial

template <typename InT, typename OutT, int D>
static cudaError_t launch_serial_typed(const void* q, const void* k, const void* v, const float* g,
                                       const float* beta, const float* S0, const int32_t* parent, int T, int B,
                                       int H, int HK, void* o, float scale, float* snap, int32_t* err,
                                       cudaStream_t st) {
    dim3 grid(D / serial::ROWS, H, B);
    serial::replay_kernel<InT, OutT, D, D><<<grid, 128, 0, st>>>(
        static_cast<const InT*>(q), static_cast<const InT*>(k), static_cast<const InT*>(v), g, beta, S0, parent,
        static_cast<OutT*>(o), snap, T, H, HK, scale, err);
    return cudaGetLastError();
}

cudaError_t launch_serial(const void* q, const void* k, const void* v, int in_bf16, const float* g,
                          const float* beta, const float* S0, const int32_t* parent, int T, int B, int H, int HK,
                          int d, void* o, int o_bf16, float scale, float* snap, int32_t* err, cudaStream_t st) {
#define CANOPY_SERIAL(IT, OT, D) \
    return launch_serial_typed<IT, OT, D>(q, k, v, g, beta, S0, parent, T, B, H, HK, o, scale, snap, err, st)
    if (d == 128) {
        if (in_bf16) {
            if (o_bf16) CANOPY_SERIAL(__nv_bfloat16, __nv_bfloat16, 128);
            CANOPY_SERIAL(__nv_bfloat16, float, 128);
        }
        if (o_bf16) CANOPY_SERIAL(float, __nv_bfloat16, 128);
        CANOPY_SERIAL(float, float, 128);
    }
    if (in_bf16) {
        if (o_bf16) CANOPY_SERIAL(__nv_bfloat16, __nv_bfloat16, 32);
        CANOPY_SERIAL(__nv_bfloat16, float, 32);
    }
    if (o_bf16) CANOPY_SERIAL(float, __nv_bfloat16, 32);
    CANOPY_SERIAL(float, float, 32);
#undef CANOPY_SERIAL
}

}  // namespace canopy
