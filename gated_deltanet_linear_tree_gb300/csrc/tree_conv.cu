// Tree-aware short causal convolution and its state commit.
//
// canopy page (projects.dotslasha.me/p/canopy.md), "M7: Benchmarks, the
// crossover, and the stretch goal": the short causal convolution (kernel 4)
// before each GDN layer follows each node's root path, and commit updates
// the convolution state with the accepted tokens.  Depthwise, per channel c:
//     y_i[c] = act(bias[c] + sum_j w[c][j] X(i, K-1-j)[c]),
// X(i, m) the input m steps up i's root path, or the committed state once
// the path has passed the root.  Memory bound: one CTA per (stream, block of
// 128 channels) stages the stream's whole block of x (T rows of 128
// channels) and its parents in shared memory in one round of coalesced
// loads.  With C a multiple of 8, one thread per node builds the node's
// table of K tap sources (a node index, or a state slot once the path has
// passed the root), and node lanes of 16 threads (eight channels each, 16-
// or 32-byte accesses) read every tap from shared memory and write y
// coalesced; otherwise node lanes of 32 threads take four channels each and
// walk the parent chain themselves.
#include "common.cuh"

namespace canopy {

namespace conv {

constexpr int NT = 256;

__device__ inline void load4c(const float* p, float (&v)[4]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ inline void load4c(const __nv_bfloat16* p, float (&v)[4]) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(w.x << 16);
    v[1] = __uint_as_float(w.x & 0xFFFF0000u);
    v[2] = __uint_as_float(w.y << 16);
    v[3] = __uint_as_float(w.y & 0xFFFF0000u);
}
// Four elements' bits, unchanged (8 bytes of bf16 or 16 of fp32).
__device__ inline void copy4c(__nv_bfloat16* d, const __nv_bfloat16* s) {
    *reinterpret_cast<uint2*>(d) = *reinterpret_cast<const uint2*>(s);
}
__device__ inline void copy4c(float* d, const float* s) {
    *reinterpret_cast<uint4*>(d) = *reinterpret_cast<const uint4*>(s);
}
__device__ inline void store4c(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ inline void store4c(__nv_bfloat16* p, const float (&v)[4]) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    *reinterpret_cast<uint2*>(p) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// The stream's parents into shared memory, sanitised as the verify does (a
// parent outside [0, i) reads as 0, the root's as -1); a bad tree is
// reported once per stream.
__device__ inline void load_parents(const int32_t* parent, int b, int T, int* sPar, int32_t* err, bool report) {
    int bad = 0;
    for (int i = threadIdx.x; i < T; i += NT) {
        int p = parent[size_t(b) * T + i];
        if (!((i == 0) ? (p == -1) : (p >= 0 && p < i))) {
            bad = CANOPY_DEVERR_TREE;
            p = (i == 0) ? -1 : 0;
        }
        sPar[i] = p;
    }
    if (bad && report && err) raise_err(err, bad);
}

constexpr int CB = 128;            // channels per CTA of the convolution
constexpr int CT = CB / 4;         // channel threads (four channels each)
constexpr int NL = NT / CT;        // node lanes

__host__ __device__ constexpr size_t conv_smem(int T, int es) { return size_t(T) * CB * es + size_t(T) * 4; }

template <typename T_, int K>
__global__ void __launch_bounds__(NT) tree_conv_kernel(const T_* __restrict__ x, const float* __restrict__ state,
                                                       const float* __restrict__ w, const float* __restrict__ bias,
                                                       const int32_t* __restrict__ parent, int T, int C, int silu,
                                                       T_* __restrict__ y, int32_t* err) {
    extern __shared__ __align__(16) uint8_t conv_smem_raw[];
    T_* sX = reinterpret_cast<T_*>(conv_smem_raw);                         // [T][CB]
    int* sPar = reinterpret_cast<int*>(conv_smem_raw + size_t(T) * CB * sizeof(T_));
    const int b = blockIdx.y, cb0 = blockIdx.x * CB;
    const int ct = threadIdx.x % CT, nl = threadIdx.x / CT;  // channel thread, node lane
    const int c = cb0 + 4 * ct;                              // first of this thread's four channels
    const bool live = c < C;
    // the stream's block of x (all rows, this CTA's channels), its parents
    // (sanitised), and this thread's weights, bias and committed state: one
    // round of independent loads
    if (live)
        for (int r = nl; r < T; r += NL) copy4c(sX + size_t(r) * CB + 4 * ct, x + (size_t(b) * T + r) * C + c);
    load_parents(parent, b, T, sPar, err, blockIdx.x == 0);
    float wv[K][4], sv[K - 1][4], bv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        bv[e] = (live && bias) ? bias[c + e] : 0.f;
#pragma unroll
        for (int j = 0; j < K; ++j) wv[j][e] = live ? w[(c + e) * K + j] : 0.f;
#pragma unroll
        for (int j = 0; j < K - 1; ++j) sv[j][e] = live ? state[(size_t(b) * C + c + e) * (K - 1) + j] : 0.f;
    }
    __syncthreads();
    if (!live) return;
    // taps m = 0 .. K-1 (weight K-1-m) walk up i's root path in shared
    // memory; once the walk has passed the root after n path nodes, tap m
    // reads the state entry K-2-(m-n), the newest first
    for (int i = nl; i < T; i += NL) {
        float acc[4] = {bv[0], bv[1], bv[2], bv[3]};
        int node = i, n = 0;
#pragma unroll
        for (int m = 0; m < K; ++m) {
            float v[4];
            if (node >= 0) {
                load4c(sX + size_t(node) * CB + 4 * ct, v);
                node = sPar[node];
                ++n;
            } else {
                const int s = K - 2 - (m - n);
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = 0.f;
#pragma unroll
                for (int ss = 0; ss < K - 1; ++ss)
                    if (ss == s)
#pragma unroll
                        for (int e = 0; e < 4; ++e) v[e] = sv[ss][e];
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] += wv[K - 1 - m][e] * v[e];
        }
        if (silu) {
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = __fdividef(acc[e], 1.f + __expf(-acc[e]));
        }
        store4c(y + (size_t(b) * T + i) * C + c, acc);
    }
}

// Eight consecutive channels (16 bytes of bf16, 32 of fp32).
__device__ inline void load8c(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        v[2 * e] = __uint_as_float(wd[e] << 16);
        v[2 * e + 1] = __uint_as_float(wd[e] & 0xFFFF0000u);
    }
}
__device__ inline void load8c(const float* p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p), c = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
}
__device__ inline void copy8c(__nv_bfloat16* d, const __nv_bfloat16* s) {
    *reinterpret_cast<uint4*>(d) = *reinterpret_cast<const uint4*>(s);
}
__device__ inline void copy8c(float* d, const float* s) {
    *reinterpret_cast<uint4*>(d) = *reinterpret_cast<const uint4*>(s);
    *reinterpret_cast<uint4*>(d + 4) = *reinterpret_cast<const uint4*>(s + 4);
}
__device__ inline void store8c(float* p, const float (&v)[8]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ inline void store8c(__nv_bfloat16* p, const float (&v)[8]) {
    uint32_t wd[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
        wd[e] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
}
// n consecutive floats (n a multiple of 4, p 16-byte aligned) into v.
template <int N>
__device__ inline void load_floats(const float* p, float (&v)[N]) {
    static_assert(N % 4 == 0, "whole float4s");
#pragma unroll
    for (int q = 0; q < N / 4; ++q) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p) + q);
        v[4 * q] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
    }
}

constexpr int CT8 = CB / 8;   // channel threads of the eight-channel kernel
constexpr int NL8 = NT / CT8; // its node lanes (two per warp)

__host__ __device__ constexpr size_t tap_offset(int T, int es) { return size_t(T) * CB * es; }
__host__ __device__ constexpr size_t par_offset(int T, int es, int K) {
    return (tap_offset(T, es) + size_t(T) * K * 2 + 15) & ~size_t(15);
}
__host__ __device__ constexpr size_t st_offset(int T, int es, int K) { return (par_offset(T, es, K) + size_t(T) * 4 + 15) & ~size_t(15); }
__host__ __device__ constexpr size_t conv8_smem(int T, int es, int K) { return st_offset(T, es, K) + size_t(K - 1) * CB * 4; }

// C a multiple of 8.  Thread i < T first lists node i's K tap sources,
// newest first: tap m is the node m steps up the root path, or, once the
// path (n nodes) has been passed, state slot K-2-(m-n), stored as -1 - slot.
template <typename T_, int K>
__global__ void __launch_bounds__(NT, (K <= 4) ? 4 : 2) tree_conv8_kernel(const T_* __restrict__ x, const float* __restrict__ state,
                                                        const float* __restrict__ w, const float* __restrict__ bias,
                                                        const int32_t* __restrict__ parent, int T, int C, int silu,
                                                        T_* __restrict__ y, int32_t* err) {
    extern __shared__ __align__(16) uint8_t conv_smem_raw[];
    T_* sX = reinterpret_cast<T_*>(conv_smem_raw);                                               // [T][CB]
    int16_t* sTap = reinterpret_cast<int16_t*>(conv_smem_raw + tap_offset(T, sizeof(T_)));       // [T][K]
    int* sPar = reinterpret_cast<int*>(conv_smem_raw + par_offset(T, sizeof(T_), K));            // [T]
    float* sS = reinterpret_cast<float*>(conv_smem_raw + st_offset(T, sizeof(T_), K));          // [K-1][CB]
    const int b = blockIdx.y, cb0 = blockIdx.x * CB;
    const int ct = threadIdx.x % CT8, nl = threadIdx.x / CT8;  // channel thread, node lane
    const int c = cb0 + 8 * ct;                                // first of this thread's eight channels
    const bool live = c < C;                                   // all eight or none (C % 8 == 0)
    // x rows four at a time, every load of a group issued before its stores
    // (one memory round trip per group rather than per row)
    constexpr int XG = 4;
    constexpr int XW = 8 * int(sizeof(T_)) / 16;  // 16-byte words per eight channels
    if (live)
        for (int r0 = nl; r0 < T; r0 += XG * NL8) {
            uint4 buf[XG][XW];
#pragma unroll
            for (int g = 0; g < XG; ++g)
                if (r0 + g * NL8 < T)
#pragma unroll
                    for (int q = 0; q < XW; ++q)
                        buf[g][q] = reinterpret_cast<const uint4*>(x + (size_t(b) * T + r0 + g * NL8) * C + c)[q];
#pragma unroll
            for (int g = 0; g < XG; ++g)
                if (r0 + g * NL8 < T)
#pragma unroll
                    for (int q = 0; q < XW; ++q)
                        reinterpret_cast<uint4*>(sX + size_t(r0 + g * NL8) * CB + 8 * ct)[q] = buf[g][q];
        }
    // the committed state of this CTA's channels (contiguous in [C][K-1]),
    // transposed to one row per slot, so that no tap waits on global memory
    {
        constexpr int SG = (CB * (K - 1) + NT - 1) / NT;
        float sv[SG];
#pragma unroll
        for (int g = 0; g < SG; ++g) {
            const int e = threadIdx.x + g * NT;
            if (e < CB * (K - 1) && cb0 + e / (K - 1) < C) sv[g] = state[(size_t(b) * C + cb0) * (K - 1) + e];
        }
#pragma unroll
        for (int g = 0; g < SG; ++g) {
            const int e = threadIdx.x + g * NT;
            if (e < CB * (K - 1) && cb0 + e / (K - 1) < C) sS[(e % (K - 1)) * CB + e / (K - 1)] = sv[g];
        }
    }
    load_parents(parent, b, T, sPar, err, blockIdx.x == 0);
    // this thread's weights (w[c .. c+7][0 .. K-1], contiguous and 16-byte
    // aligned since c is a multiple of 8) and bias; the committed state is
    // read only by the few nodes within K - 1 steps of the root
    float wf[8 * K], bv[8];
    if (live) {
        load_floats(w + size_t(c) * K, wf);
#pragma unroll
        for (int e = 0; e < 8; ++e) bv[e] = bias ? bias[c + e] : 0.f;  // bias is only 4-byte aligned
    }
    __syncthreads();
    if (threadIdx.x < T) {
        const int i = threadIdx.x;
        int node = i, n = 0;
#pragma unroll
        for (int m = 0; m < K; ++m) {
            int tap;
            if (node >= 0) {
                tap = node;
                node = sPar[node];
                ++n;
            } else {
                tap = -1 - (K - 2 - (m - n));
            }
            sTap[i * K + m] = int16_t(tap);
        }
    }
    __syncthreads();
    if (!live) return;
    for (int i = nl; i < T; i += NL8) {
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = bv[e];
#pragma unroll
        for (int m = 0; m < K; ++m) {
            const int t = sTap[i * K + m];
            float v[8];
            if (t >= 0) {
                load8c(sX + size_t(t) * CB + 8 * ct, v);
            } else {
                const float4* sp = reinterpret_cast<const float4*>(sS + (-1 - t) * CB + 8 * ct);
                const float4 a0 = sp[0], a1 = sp[1];
                v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w;
                v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(wf[e * K + (K - 1 - m)], v[e], acc[e]);
        }
        if (silu) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = __fdividef(acc[e], 1.f + __expf(-acc[e]));
        }
        store8c(y + (size_t(b) * T + i) * C + c, acc);
    }
}

template <typename T_, int K>
__global__ void __launch_bounds__(NT) conv_commit_kernel(const int32_t* __restrict__ accepted, const T_* __restrict__ x,
                                                         const int32_t* __restrict__ parent, const float* state,
                                                         float* state_new, int T, int C, int32_t* err) {
    __shared__ int sPar[kMaxT];
    const int b = blockIdx.y;
    const int c0 = 4 * (blockIdx.x * NT + threadIdx.x);
    load_parents(parent, b, T, sPar, nullptr, false);
    __syncthreads();
    if (c0 >= C) return;
    int a = accepted[b];
    if (a < -1 || a >= T) {
        if (err && c0 == 0) raise_err(err, CANOPY_DEVERR_ACCEPTED);
        a = -1;
    }
    float old[K - 1][4], nw[K - 1][4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int j = 0; j < K - 1; ++j) old[j][e] = state[(size_t(b) * C + c0 + e) * (K - 1) + j];
    // newest first (position K - 2 - m): the accepted path from a up to the
    // root, then the old state from its newest entry
    int node = a, n = 0;  // n: path nodes used
#pragma unroll
    for (int m = 0; m < K - 1; ++m) {
        if (node >= 0) {
            float v[4];
            load4c(x + (size_t(b) * T + node) * C + c0, v);
#pragma unroll
            for (int e = 0; e < 4; ++e) nw[K - 2 - m][e] = v[e];
            node = sPar[node];
            ++n;
        } else {
            const int s = K - 2 - (m - n);
#pragma unroll
            for (int ss = 0; ss < K - 1; ++ss)
                if (ss == s)
#pragma unroll
                    for (int e = 0; e < 4; ++e) nw[K - 2 - m][e] = old[ss][e];
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int j = 0; j < K - 1; ++j) state_new[(size_t(b) * C + c0 + e) * (K - 1) + j] = nw[j][e];
}

}  // namespace conv

template <typename T_, int K>
static cudaError_t tree_conv_typed(dim3 grid, const void* x, const float* state, const float* w, const float* bias,
                                   const int32_t* parent, int T, int C, int silu, void* y, int32_t* err,
                                   cudaStream_t st) {
    if (C % 8 == 0) {
        static bool attr8 = false;
        if (!attr8) {
            const cudaError_t e = cudaFuncSetAttribute(conv::tree_conv8_kernel<T_, K>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       int(conv::conv8_smem(kMaxT, sizeof(T_), K)));
            if (e != cudaSuccess) return e;
            attr8 = true;
        }
        conv::tree_conv8_kernel<T_, K><<<grid, conv::NT, conv::conv8_smem(T, sizeof(T_), K), st>>>(
            static_cast<const T_*>(x), state, w, bias, parent, T, C, silu, static_cast<T_*>(y), err);
        return cudaGetLastError();
    }
    static bool attr = false;
    if (!attr) {
        const cudaError_t e = cudaFuncSetAttribute(conv::tree_conv_kernel<T_, K>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   int(conv::conv_smem(kMaxT, sizeof(T_))));
        if (e != cudaSuccess) return e;
        attr = true;
    }
    conv::tree_conv_kernel<T_, K><<<grid, conv::NT, conv::conv_smem(T, sizeof(T_)), st>>>(
        static_cast<const T_*>(x), state, w, bias, parent, T, C, silu, static_cast<T_*>(y), err);
    return cudaGetLastError();
}

template <typename T_, int K>
static void conv_commit_typed(dim3 grid, const int32_t* accepted, const void* x, const int32_t* parent,
                              const float* state, float* state_new, int T, int C, int32_t* err, cudaStream_t st) {
    conv::conv_commit_kernel<T_, K><<<grid, conv::NT, 0, st>>>(accepted, static_cast<const T_*>(x), parent, state,
                                                              state_new, T, C, err);
}

cudaError_t launch_tree_conv(const void* x, int bf16, const float* state, const float* w, const float* bias,
                             const int32_t* parent, int T, int B, int C, int K, int silu, void* y, int32_t* err,
                             cudaStream_t st) {
    dim3 grid((C + conv::CB - 1) / conv::CB, B);
#define CANOPY_CONV(KK)                                                                                        \
    case KK:                                                                                                   \
        return bf16 ? tree_conv_typed<__nv_bfloat16, KK>(grid, x, state, w, bias, parent, T, C, silu, y, err, st) \
                    : tree_conv_typed<float, KK>(grid, x, state, w, bias, parent, T, C, silu, y, err, st);
    switch (K) {
        CANOPY_CONV(2) CANOPY_CONV(3) CANOPY_CONV(4) CANOPY_CONV(5) CANOPY_CONV(6) CANOPY_CONV(7) CANOPY_CONV(8)
        default: return cudaErrorInvalidValue;
    }
#undef CANOPY_CONV
}

cudaError_t launch_conv_commit(const int32_t* accepted, const void* x, int bf16, const int32_t* parent,
                               const float* state, float* state_new, int T, int B, int C, int K, int32_t* err,
                               cudaStream_t st) {
    dim3 grid((C / 4 + conv::NT - 1) / conv::NT, B);
#define CANOPY_CCOMMIT(KK)                                                                                \
    case KK:                                                                                              \
        if (bf16)                                                                                         \
            conv_commit_typed<__nv_bfloat16, KK>(grid, accepted, x, parent, state, state_new, T, C, err, st); \
        else                                                                                              \
            conv_commit_typed<float, KK>(grid, accepted, x, parent, state, state_new, T, C, err, st);         \
        break;
    switch (K) {
        CANOPY_CCOMMIT(2) CANOPY_CCOMMIT(3) CANOPY_CCOMMIT(4) CANOPY_CCOMMIT(5) CANOPY_CCOMMIT(6)
        CANOPY_CCOMMIT(7) CANOPY_CCOMMIT(8)
        default: return cudaErrorInvalidValue;
    }
#undef CANOPY_CCOMMIT
    return cudaGetLastError();
}

}  // namespace canopy
