// Solve variants of the tree verify beside the blocked substitution: the
// finite Neumann series, the squaring form and the split design.
//
// canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed form":
// G is nilpotent (G^(d+1) = 0 for a tree of depth d), so
//     (I + G)^-1 = sum_{m=0..d} (-G)^m                      (Neumann series)
//                = (I - G)(I + G^2)(I + G^4) ... (I + G^(2^(k-1))),
// with k = ceil(log2(d + 1)) factors (the squaring form); and "Design
// decisions" (the split alternative: (I + G)^-1 built once per (stream,
// value head) in global memory, then applied per value tile).
//
// All three start from the tensor-core Gram's scratch (gram_tc.cu): G and C
// as [B][H][T][T] (64 x 64 tiles on and below the diagonal, zero off the
// paths), gamma X_Q and R as [B][T][H][dv]; like the blocked substitution
// they write U = (I + G)^-1 R to the workspace (the commit reads it) and
//     o = scale (gamma X_Q + C U).
// The Neumann series beyond 64 nodes and the squaring form run on tensor
// cores (neumann_tc.cu, squaring_tc.cu); the split design's two kernels here
// are fp32 on CUDA cores, 64 x 64 tiles through shared memory:
//   invert_kernel   one CTA per (stream, head): W = (I + G)^-1 in place of G
//                   (block row by block row) and M = C W in place of C;
//   apply_kernel    one CTA per (stream, head, 64-node block, 64 value
//                   columns): U_r = sum_s W_rs R_s, o_r = gamma X_Q,r +
//                   sum_s M_rs R_s, with no dependence between CTAs.
// The split kernels overwrite the G and C scratch (and the squaring form G),
// which nothing reads after the verify.
#include <algorithm>

#include "common.cuh"

namespace canopy {

namespace sv {

constexpr int BN = 64;    // nodes per tile
constexpr int GS = 68;    // row stride of a staged tile (floats)
constexpr int DV = 128;   // value columns (dk = dv = 128)
constexpr int NT = 512;   // threads of the per-(stream, head) kernels
constexpr int APPLY_NT = 256;

// Tile (r, s) of a [T][T] matrix into a [BN][GS] staging tile; entries
// outside the tree (row or column >= T) read as zero.  The matrix may have
// been written earlier in the same kernel, so no read-only path is used.
__device__ __forceinline__ void load_tile(float* dst, const float* m, int T, int r, int s, int t, int nt) {
    const int i0 = BN * r, j0 = BN * s;
    if ((T & 3) == 0) {
        for (int e = t; e < BN * BN / 4; e += nt) {
            const int rho = e >> 4, j = (e & 15) * 4, i = i0 + rho, jj = j0 + j;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < T && jj < T) x = *reinterpret_cast<const float4*>(m + size_t(i) * T + jj);
            *reinterpret_cast<float4*>(dst + rho * GS + j) = x;
        }
    } else {
        for (int e = t; e < BN * BN; e += nt) {
            const int rho = e >> 6, j = e & 63, i = i0 + rho, jj = j0 + j;
            dst[rho * GS + j] = (i < T && jj < T) ? m[size_t(i) * T + jj] : 0.f;
        }
    }
}

// A [BN][GS] tile from registers back to tile (r, s) of a [T][T] matrix:
// rows 4 rg .. 4 rg + MR - 1 (MR of them), columns 4 cg .. 4 cg + 3.
template <int MR>
__device__ __forceinline__ void store_tile_part(float* m, int T, int r, int s, int row0, int col0,
                                                const float (&acc)[MR][4]) {
#pragma unroll
    for (int q = 0; q < MR; ++q) {
        const int i = BN * r + row0 + q;
        if (i >= T) continue;
        float* p = m + size_t(i) * T + BN * s + col0;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
            if (BN * s + col0 + cc < T) p[cc] = acc[q][cc];
    }
}

// acc[q][c] (+/-)= sum_{k<64} A[q][k] B[k][c], q < MR, c < 4; A rows at
// stride GS, B rows at stride BS (a and b already offset to the thread's
// rows and columns).
template <int MR, int BS, bool SUB>
__device__ __forceinline__ void mac(float (&acc)[MR][4], const float* a, const float* b) {
#pragma unroll 2
    for (int k = 0; k < BN; k += 4) {
        float4 u[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) u[kk] = *reinterpret_cast<const float4*>(b + (k + kk) * BS);
#pragma unroll
        for (int q = 0; q < MR; ++q) {
            const float4 w = *reinterpret_cast<const float4*>(a + q * GS + k);
            const float x = (w.x * u[0].x + w.y * u[1].x) + (w.z * u[2].x + w.w * u[3].x);
            const float y = (w.x * u[0].y + w.y * u[1].y) + (w.z * u[2].y + w.w * u[3].y);
            const float z = (w.x * u[0].z + w.y * u[1].z) + (w.z * u[2].z + w.w * u[3].z);
            const float v = (w.x * u[0].w + w.y * u[1].w) + (w.z * u[2].w + w.w * u[3].w);
            if (SUB) {
                acc[q][0] -= x; acc[q][1] -= y; acc[q][2] -= z; acc[q][3] -= v;
            } else {
                acc[q][0] += x; acc[q][1] += y; acc[q][2] += z; acc[q][3] += v;
            }
        }
    }
}

// Split design, first kernel: W = (I + G)^-1 and M = C W per (stream,
// head), in place of G and C, block row by block row from the top.
//   W_rr = (I + G_rr)^-1: row rho along its in-block path (nodes of block r
//     on path(rho), root side first, rho last), from rho up:
//     W[rho][rho] = 1, W[rho][k] = -sum_{e below k on the path} W[rho][e] G[e][k];
//   W_rc = -W_rr sum_{s=c..r-1} G_rs W_sc for c < r, from left to right (the
//     old G_rc is read by no later tile of the row);
//   M_rc = sum_{s=c..r} C_rs W_sc for c <= r, from left to right.
__global__ void __launch_bounds__(NT, 1) invert_kernel(int T, int H, Ws ws) {
    extern __shared__ float smem[];
    float* sA = smem;              // [BN][GS]
    float* sB = sA + BN * GS;      // [BN][GS]
    float* sW = sB + BN * GS;      // [BN][GS] W_rr
    float* sS = sW + BN * GS;      // [BN][GS] staged partial sums
    uint8_t* sPl = reinterpret_cast<uint8_t*>(sS + BN * GS);  // [BN][BN] in-block paths
    const int h = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
    const int cg = t & 15, rg = t >> 4;  // 2 x 4 entries of a 64 x 64 tile per thread
    const size_t bh = size_t(b) * H + h;
    float* W = ws.gs + bh * T * T;   // G on entry, W on exit
    float* M = ws.cs + bh * T * T;   // C on entry, M on exit
    const int nb = (T + BN - 1) / BN;

    for (int r = 0; r < nb; ++r) {
        __syncthreads();
        load_tile(sA, W, T, r, r, t, NT);  // G_rr (row r is still G)
        if (t < BN) {
            const int rho = t, i = BN * r + rho;
            uint64_t bits = 0;
            if (i < T) {
                const uint32_t* mrow = ws.mask + (size_t(b) * T + i) * ws.W;
                const uint32_t w0 = mrow[2 * r], w1 = (2 * r + 1 < ws.W) ? mrow[2 * r + 1] : 0u;
                bits = (uint64_t(w1) << 32 | w0) | (1ull << rho);
            }
            int n = 0;
            for (; bits; bits &= bits - 1) sPl[rho * BN + n++] = uint8_t(__ffsll(static_cast<long long>(bits)) - 1);
            for (int z = n; z < BN; ++z) sPl[rho * BN + z] = 0xFF;
        }
        __syncthreads();
        if (t < BN) {
            const int rho = t;
            const uint8_t* pl = sPl + rho * BN;
            float* wr = sW + rho * GS;
            for (int j = 0; j < BN; ++j) wr[j] = 0.f;
            int n = 0;
            while (n < BN && pl[n] != 0xFF) ++n;
            // rows past T have the empty path: a zero row
            if (BN * r + rho < T) {
                for (int e = n - 1; e >= 0; --e) {
                    const int kcol = pl[e];
                    float acc = (e == n - 1) ? 1.f : 0.f;
                    for (int f = e + 1; f < n; ++f) acc -= wr[pl[f]] * sA[pl[f] * GS + kcol];
                    wr[kcol] = acc;
                }
            }
        }
        // W_rc for c < r (its sum needs W_sc of rows above, already inverted)
        for (int c = 0; c < r; ++c) {
            float acc[2][4] = {};
            for (int s = c; s < r; ++s) {
                __syncthreads();
                load_tile(sA, W, T, r, s, t, NT);  // G_rs: row r is overwritten only left of c
                load_tile(sB, W, T, s, c, t, NT);  // W_sc
                __syncthreads();
                mac<2, GS, false>(acc, sA + 2 * rg * GS, sB + 4 * cg);
            }
#pragma unroll
            for (int q = 0; q < 2; ++q)
                *reinterpret_cast<float4*>(sS + (2 * rg + q) * GS + 4 * cg) =
                    make_float4(acc[q][0], acc[q][1], acc[q][2], acc[q][3]);
            __syncthreads();
            float w[2][4] = {};
            mac<2, GS, true>(w, sW + 2 * rg * GS, sS + 4 * cg);
            store_tile_part<2>(W, T, r, c, 2 * rg, 4 * cg, w);
        }
        __syncthreads();
        {
            float w[2][4];
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) w[q][cc] = sW[(2 * rg + q) * GS + 4 * cg + cc];
            store_tile_part<2>(W, T, r, r, 2 * rg, 4 * cg, w);
        }
        // M_rc = sum_{s=c..r} C_rs W_sc (row r of W is complete)
        for (int c = 0; c <= r; ++c) {
            float acc[2][4] = {};
            for (int s = c; s <= r; ++s) {
                __syncthreads();  // also orders the W (and M) stores above before these loads
                load_tile(sA, M, T, r, s, t, NT);  // C_rs: row r of M is overwritten only left of c
                load_tile(sB, W, T, s, c, t, NT);
                __syncthreads();
                mac<2, GS, false>(acc, sA + 2 * rg * GS, sB + 4 * cg);
            }
            store_tile_part<2>(M, T, r, c, 2 * rg, 4 * cg, acc);
        }
    }
}

// Split design, second kernel: per (stream, head, block r, 64 value
// columns) U_r = sum_{s<=r} W_rs R_s and o_r = scale (gamma X_Q,r +
// sum_{s<=r} M_rs R_s).  4 x 4 entries per thread.
template <typename OutT>
__global__ void __launch_bounds__(APPLY_NT) apply_kernel(OutT* __restrict__ o, int T, int H, Ws ws, float scale) {
    extern __shared__ float smem[];
    float* sA = smem;            // [BN][GS] W_rs
    float* sB = sA + BN * GS;    // [BN][GS] M_rs
    float* sR = sB + BN * GS;    // [BN][BN] R_s, this CTA's value columns
    const int r = blockIdx.x >> 1, half = blockIdx.x & 1, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
    const int cg = t & 15, rg = t >> 4;
    const int col0 = BN * half;
    const size_t bh = size_t(b) * H + h;
    const float* W = ws.gs + bh * T * T;
    const float* M = ws.cs + bh * T * T;
    float u[4][4] = {}, acc[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int i = BN * r + 4 * rg + q;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < T) x = *reinterpret_cast<const float4*>(ws.xq + ((size_t(b) * T + i) * H + h) * DV + col0 + 4 * cg);
        acc[q][0] = x.x; acc[q][1] = x.y; acc[q][2] = x.z; acc[q][3] = x.w;
    }
    for (int s = 0; s <= r; ++s) {
        __syncthreads();
        load_tile(sA, W, T, r, s, t, APPLY_NT);
        load_tile(sB, M, T, r, s, t, APPLY_NT);
        for (int e = t; e < BN * BN / 4; e += APPLY_NT) {
            const int j = e >> 4, c4 = e & 15, i = BN * s + j;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < T) x = *reinterpret_cast<const float4*>(ws.rr + ((size_t(b) * T + i) * H + h) * DV + col0 + 4 * c4);
            *reinterpret_cast<float4*>(sR + j * BN + 4 * c4) = x;
        }
        __syncthreads();
        mac<4, BN, false>(u, sA + 4 * rg * GS, sR + 4 * cg);
        mac<4, BN, false>(acc, sB + 4 * rg * GS, sR + 4 * cg);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int i = BN * r + 4 * rg + q;
        if (i >= T) continue;
        const size_t ni = (size_t(b) * T + i) * H + h;
        *reinterpret_cast<float4*>(ws.U + ni * DV + col0 + 4 * cg) = make_float4(u[q][0], u[q][1], u[q][2], u[q][3]);
        OutT* op = o + ni * DV + col0 + 4 * cg;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) store_out(op + cc, scale * acc[q][cc]);
    }
}

constexpr size_t kInvertSmem = size_t(4) * BN * GS * 4 + size_t(BN) * BN;
constexpr size_t kApplySmem = size_t(2) * BN * GS * 4 + size_t(BN) * BN * 4;

}  // namespace sv

// ---------------------------------------------------------------------------
// Host side.  The Gram scratch must be in place (launch_gram_tc).

template <typename K>
static cudaError_t set_smem_once(K kernel, size_t bytes, bool& done) {
    if (done) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
    if (e == cudaSuccess) done = true;
    return e;
}

template <typename OutT>
static cudaError_t launch_variant_typed(int variant, int T, int B, int H, OutT* o, float scale, const Ws& ws,
                                        cudaStream_t st) {
    dim3 grid(H, B);
    cudaError_t e;
    if (variant == 3) {
        static bool attr = false;
        e = set_smem_once(sv::invert_kernel, sv::kInvertSmem, attr);
        if (e != cudaSuccess) return e;
        sv::invert_kernel<<<grid, sv::NT, sv::kInvertSmem, st>>>(T, H, ws);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        static bool attr2 = false;
        e = set_smem_once(sv::apply_kernel<OutT>, sv::kApplySmem, attr2);
        if (e != cudaSuccess) return e;
        dim3 g2(2 * ((T + sv::BN - 1) / sv::BN), H, B);
        sv::apply_kernel<OutT><<<g2, sv::APPLY_NT, sv::kApplySmem, st>>>(o, T, H, ws, scale);
        return cudaGetLastError();
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_neumann_tc(int T, int B, int H, void* o, int o_bf16, float scale, const Ws& ws, cudaStream_t st);
cudaError_t launch_squaring_tc(int T, int B, int H, void* o, int o_bf16, float scale, const Ws& ws, cudaStream_t st);

// variant: 1 Neumann series (on tensor cores, neumann_tc.cu; T > 64), 2
// squaring form (on tensor cores, squaring_tc.cu), 3 split design (dk = dv =
// 128).
cudaError_t launch_solve_variant(int variant, int T, int B, int H, void* o, int o_bf16, float scale, const Ws& ws,
                                 cudaStream_t st) {
    if (T < 1 || T > kMaxT) return cudaErrorInvalidValue;
    if (variant == 1) return launch_neumann_tc(T, B, H, o, o_bf16, scale, ws, st);
    if (variant == 2) return launch_squaring_tc(T, B, H, o, o_bf16, scale, ws, st);
    if (o_bf16)
        return launch_variant_typed(variant, T, B, H, static_cast<__nv_bfloat16*>(o), scale, ws, st);
    return launch_variant_typed(variant, T, B, H, static_cast<float*>(o), scale, ws, st);
}

}  // namespace canopy
